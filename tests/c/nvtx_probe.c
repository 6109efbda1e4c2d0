/* A minimal NVTX tool for the host tests: loaded through NVTX_INJECTION64_PATH,
 * it replaces the range push / pop callbacks with functions that record each
 * range's name and the nesting depth, which the test reads back through
 * nvtx_probe_log().  No GPU is involved: the ranges wrap the library's C-ABI
 * calls, including calls that fail their argument checks. */
#include <string.h>

#include <nvtx3/nvToolsExt.h>

static char g_log[8192];
static size_t g_len;
static int g_depth;

static void append(const char *s) {
  size_t n = strlen(s);
  if (g_len + n + 1 >= sizeof g_log) return;
  memcpy(g_log + g_len, s, n);
  g_len += n;
  g_log[g_len] = 0;
}

static int probe_push(const char *message) {
  append("+");
  append(message ? message : "?");
  append(";");
  return g_depth++;
}

static int probe_pop(void) {
  append("-;");
  return --g_depth;
}

/* Called by NVTX on the first range call of the process. */
__attribute__((visibility("default"))) int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get) {
  const NvtxExportTableCallbacks *cb =
      (const NvtxExportTableCallbacks *)get(NVTX_ETID_CALLBACKS);
  NvtxFunctionTable table = 0;
  unsigned int size = 0;
  if (!cb || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &size)) return 0;
  if (size <= NVTX_CBID_CORE_RangePop) return 0;
  *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)probe_push;
  *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)probe_pop;
  return 1;
}

/* "+name;" for each push and "-;" for each pop, in call order. */
__attribute__((visibility("default"))) const char *nvtx_probe_log(void) { return g_log; }
