/* The public header as a plain C (C11) program: librpa's C ABI used from C,
 * with no GPU: plan a small ragged batch on the host, read the plan's info,
 * check a status string and an argument error.  Built and run by the test
 * suite; prints one line and returns 0 on success. */
#include <stdio.h>
#include <string.h>

#include "rpa.h"

int main(void) {
  const int32_t cu[4] = {0, 1, 2, 40};      /* two decode tokens, a 38-token chunk */
  const int32_t kv[3] = {100, 300, 500};
  rpa_plan_options o;
  memset(&o, 0, sizeof(o));
  o.struct_size = (int32_t)sizeof(o);
  o.num_sms = 152;
  rpa_plan_t* plan = NULL;
  size_t ws = 0;
  rpa_status_t st = rpa_plan(&plan, cu, kv, NULL, 3, 8, 2, 128, 16, 32, 64, RPA_DTYPE_BF16, &o, &ws);
  if (st != RPA_OK) { printf("rpa_plan: %s\n", rpa_status_string(st)); return 1; }
  rpa_plan_info info;
  memset(&info, 0, sizeof(info));
  if (rpa_plan_get_info(plan, &info) != RPA_OK) return 2;
  if (info.num_decode_seqs != 2 || info.num_prefill_seqs != 1 || info.workspace_bytes != (int64_t)ws)
    return 3;
  if (rpa_plan_destroy(plan) != RPA_OK) return 4;
  /* A q-head count that is not a multiple of the KV heads is refused on the host. */
  plan = NULL;
  st = rpa_plan(&plan, cu, kv, NULL, 3, 6, 4, 128, 16, 32, 64, RPA_DTYPE_BF16, &o, &ws);
  if (st != RPA_ERR_INVALID_ARG || plan != NULL) return 5;
  if (strncmp(rpa_status_string(RPA_ERR_PLAN_MISMATCH), "RPA_", 4) != 0) return 6;
  printf("c abi ok: path %d, %d decode, %d prefill items, workspace %lld bytes\n", info.path,
         info.num_decode_seqs, info.num_prefill_items, (long long)info.workspace_bytes);
  return 0;
}
