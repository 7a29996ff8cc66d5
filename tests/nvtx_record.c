/* A minimal NVTX tool for the tests: loaded by the NVTX runtime through
 * NVTX_INJECTION64_PATH, it replaces the domain create, range push and range
 * pop callbacks with recorders and exposes what they saw as text, one event
 * per line ("domain <name>", "push <domain> <message>", "pop <domain>"). */
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static char log_buf[8192];
#define DOMAIN ((nvtxDomainHandle_t)(uintptr_t)0x1234)

static void note(const char* s) {
    size_t n = strlen(log_buf), m = strlen(s);
    if (n + m + 2 < sizeof log_buf) {
        memcpy(log_buf + n, s, m);
        log_buf[n + m] = '\n';
        log_buf[n + m + 1] = 0;
    }
}
static nvtxDomainHandle_t create_a(const char* name) {
    char b[256];
    snprintf(b, sizeof b, "domain %s", name);
    note(b);
    return DOMAIN;
}
static int push_ex(nvtxDomainHandle_t d, const nvtxEventAttributes_t* a) {
    char b[256];
    snprintf(b, sizeof b, "push %s %s", d == DOMAIN ? "pagedkv" : "?",
             a->messageType == NVTX_MESSAGE_TYPE_ASCII ? a->message.ascii : "?");
    note(b);
    return 0;
}
static int pop(nvtxDomainHandle_t d) {
    note(d == DOMAIN ? "pop pagedkv" : "pop ?");
    return 0;
}
int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get) {
    const NvtxExportTableCallbacks* cb = (const NvtxExportTableCallbacks*)get(NVTX_ETID_CALLBACKS);
    NvtxFunctionTable t = 0;
    unsigned int n = 0;
    if (!cb || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE2, &t, &n)) return 0;
    if (n <= NVTX_CBID_CORE2_DomainCreateA) return 0;
    *t[NVTX_CBID_CORE2_DomainCreateA] = (NvtxFunctionPointer)create_a;
    *t[NVTX_CBID_CORE2_DomainRangePushEx] = (NvtxFunctionPointer)push_ex;
    *t[NVTX_CBID_CORE2_DomainRangePop] = (NvtxFunctionPointer)pop;
    return 1;
}
const char* injection_log(void) { return log_buf; }
