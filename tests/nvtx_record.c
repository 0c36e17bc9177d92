/* A minimal NVTX v3 tool for the tests: NVTX loads it from the path in
 * NVTX_INJECTION64_PATH and calls InitializeInjectionNvtx2, which points the
 * domain-create, range-push and range-pop entries of NVTX's callback table at
 * functions that append one line per event to the file named by
 * TP_NVTX_RECORD ("domain <name>", "push <message>", "pop"). */
#include <stdio.h>
#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

static FILE* g_out;

static nvtxDomainHandle_t NVTX_API rec_domain_create(const char* name) {
  fprintf(g_out, "domain %s\n", name);
  fflush(g_out);
  return (nvtxDomainHandle_t)&g_out;
}

static int NVTX_API rec_push(nvtxDomainHandle_t domain, const nvtxEventAttributes_t* a) {
  (void)domain;
  fprintf(g_out, "push %s\n", (a && a->messageType == NVTX_MESSAGE_TYPE_ASCII) ? a->message.ascii : "?");
  fflush(g_out);
  return 0;
}

static int NVTX_API rec_pop(nvtxDomainHandle_t domain) {
  (void)domain;
  fprintf(g_out, "pop\n");
  fflush(g_out);
  return 0;
}

int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_table) {
  const char* path = getenv("TP_NVTX_RECORD");
  if (!path || !(g_out = fopen(path, "w"))) return 0;
  const NvtxExportTableCallbacks* cb = (const NvtxExportTableCallbacks*)get_table(NVTX_ETID_CALLBACKS);
  NvtxFunctionTable table = 0;
  unsigned int size = 0;
  if (!cb || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE2, &table, &size) || !table) return 0;
  if (size <= NVTX_CBID_CORE2_DomainCreateA) return 0;
  *table[NVTX_CBID_CORE2_DomainCreateA] = (NvtxFunctionPointer)rec_domain_create;
  *table[NVTX_CBID_CORE2_DomainRangePushEx] = (NvtxFunctionPointer)rec_push;
  *table[NVTX_CBID_CORE2_DomainRangePop] = (NvtxFunctionPointer)rec_pop;
  return 1;
}
