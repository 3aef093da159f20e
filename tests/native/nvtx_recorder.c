/*
 * nvtx_recorder.c -- a minimal NVTX injection library for the CPU tests.
 *
 * NVTX calls in a program do nothing until a tool attaches: at the first
 * call, the NVTX runtime loads the library named by NVTX_INJECTION64_PATH
 * and calls its InitializeInjectionNvtx2, which may fill in the slots of the
 * core function table.  This one records every nvtxRangePushA message and
 * counts the pops, so a test can check which ranges a C-ABI call opened and
 * that it closed them.  It links to nothing of the library under test.
 */
#include <stdint.h>
#include <string.h>

#include "nvtx3/nvToolsExt.h"

static char g_names[1 << 16];
static size_t g_len;
static int g_depth, g_pops;

static int NVTX_API record_push(const char* message) {
    const size_t n = strlen(message);
    if (g_len + n + 2 < sizeof g_names) {
        memcpy(g_names + g_len, message, n);
        g_len += n;
        g_names[g_len++] = '\n';
        g_names[g_len] = 0;
    }
    return g_depth++;
}

static int NVTX_API record_pop(void) {
    ++g_pops;
    return --g_depth;
}

int NVTX_API InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_export_table) {
    const NvtxExportTableCallbacks* cb =
        (const NvtxExportTableCallbacks*)get_export_table(NVTX_ETID_CALLBACKS);
    NvtxFunctionTable table = 0;
    unsigned int size = 0;
    if (!cb || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &size)) return 0;
    if (size < NVTX_CBID_CORE_RangePop) return 0;
    *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)record_push;
    *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)record_pop;
    return 1;
}

const char* recorded_names(void) { return g_names; }
int recorded_pops(void) { return g_pops; }
int recorded_depth(void) { return g_depth; }
