// Library-wide utilities of the C ABI: status strings, error-word check,
// bounded-wait limit, launch accounting, device properties cache.
#include <atomic>
#include <mutex>

#include "fs_common.cuh"

namespace fs {
namespace {
std::atomic<int64_t> g_launches{0};
std::atomic<int64_t> g_spin_limit{int64_t(1) << 22};
std::atomic<int64_t> g_skip_tile{-1};
std::mutex g_sm_mu;
int g_sm_count[64] = {0};
}  // namespace

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  std::lock_guard<std::mutex> lk(g_sm_mu);
  if (g_sm_count[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 152;
    g_sm_count[dev] = v;
  }
  return g_sm_count[dev];
}

int64_t spin_limit() { return g_spin_limit.load(); }
int64_t debug_skip_tile() { return g_skip_tile.load(); }
void count_launch(int k) { g_launches.fetch_add(k); }

}  // namespace fs

extern "C" fs_status fs_check(const int32_t* err, fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FS_ERR_CUDA;
  if (!err) return FS_OK;
  int32_t v = 0;
  if (cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return FS_ERR_CUDA;
  return static_cast<fs_status>(v);
}

extern "C" const char* fs_status_string(fs_status s) {
  switch (s) {
    case FS_OK: return "ok";
    case FS_ERR_INVALID_ARG: return "invalid argument";
    case FS_ERR_ID_RANGE: return "ID outside [0, num_rows)";
    case FS_ERR_BAD_OFFSETS: return "malformed offsets or permutation";
    case FS_ERR_CAPACITY: return "output capacity exceeded";
    case FS_ERR_WORKSPACE: return "workspace too small";
    case FS_ERR_TIMEOUT: return "bounded inter-block wait gave up";
    case FS_ERR_CUDA: return "CUDA runtime error";
    case FS_ERR_ALIGNMENT: return "misaligned pointer";
  }
  return "unknown status";
}

extern "C" void fs_set_spin_limit(int64_t polls) { fs::g_spin_limit.store(polls < 1 ? 1 : polls); }

extern "C" int64_t fs_get_spin_limit(void) { return fs::g_spin_limit.load(); }

extern "C" void fs_debug_skip_publish(int64_t tile) { fs::g_skip_tile.store(tile); }

extern "C" int64_t fs_launch_count(void) { return fs::g_launches.load(); }

extern "C" const char* fs_version(void) { return "fsjagged 0.1 (sm_103a)"; }
