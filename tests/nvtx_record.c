/* NVTX injection library for tests: records every range push and pop of the process to
 * the file named by SSM_NVTX_LOG, one line each ("push <name>" / "pop").  Loaded by the
 * NVTX3 headers' own loader when NVTX_INJECTION64_PATH names this library; it fills the
 * core module's RangePushA and RangePop slots through the export table the loader hands
 * to InitializeInjectionNvtx2. */
#include <stdio.h>
#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

static FILE* g_out;

static int NVTX_API record_push(const char* message) {
    fprintf(g_out, "push %s\n", message ? message : "");
    fflush(g_out);
    return 0;
}

static int NVTX_API record_pop(void) {
    fprintf(g_out, "pop\n");
    fflush(g_out);
    return 0;
}

int NVTX_API InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_export_table) {
    const NvtxExportTableCallbacks* cb = (const NvtxExportTableCallbacks*)get_export_table(NVTX_ETID_CALLBACKS);
    NvtxFunctionTable table = 0;
    unsigned int size = 0;
    const char* path = getenv("SSM_NVTX_LOG");
    if (!cb || !path || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &size)) return 0;
    if (size <= NVTX_CBID_CORE_RangePop || size <= NVTX_CBID_CORE_RangePushA) return 0;
    g_out = fopen(path, "w");
    if (!g_out) return 0;
    *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)record_push;
    *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)record_pop;
    return 1;
}
