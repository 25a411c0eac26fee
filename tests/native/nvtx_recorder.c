/*
 * NVTX injection library used by the CPU tests: it records the NVTX ranges a
 * process opens and closes, one line per event, in the file named by the
 * FS_NVTX_LOG environment variable.  A process loads it when
 * NVTX_INJECTION64_PATH points at it; the NVTX runtime then calls
 * InitializeInjectionNvtx2, which installs the two recorders below in the
 * core module's callback table (push of a named range, pop).
 */
#include <stdio.h>
#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

static FILE* g_log = NULL;

static int NVTX_API record_push(const char* name) {
  if (g_log) {
    fprintf(g_log, "push %s\n", name ? name : "");
    fflush(g_log);
  }
  return 0;
}

static int NVTX_API record_pop(void) {
  if (g_log) {
    fputs("pop\n", g_log);
    fflush(g_log);
  }
  return 0;
}

int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_table) {
  const NvtxExportTableCallbacks* cb = (const NvtxExportTableCallbacks*)get_table(NVTX_ETID_CALLBACKS);
  NvtxFunctionTable table = NULL;
  unsigned int slots = 0;
  const char* path = getenv("FS_NVTX_LOG");
  if (!cb || !path || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &slots)) return 0;
  if (slots <= NVTX_CBID_CORE_RangePop) return 0;
  g_log = fopen(path, "w");
  if (!g_log) return 0;
  *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)record_push;
  *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)record_pop;
  return 1;
}
