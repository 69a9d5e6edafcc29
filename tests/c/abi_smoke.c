/* Plain C99 use of include/vc.h: the header compiles as C, the library links,
 * and the host-only entry points answer without a GPU. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "vc.h"

int main(void) {
  if (strcmp(vc_status_string(VC_ERR_UNSUPPORTED), "VC_ERR_UNSUPPORTED") != 0) return 1;
  if (vc_busbw_factor(VC_COLL_ALLREDUCE, 8) != 1.75) return 2;
  size_t n = 0, scratch = 0;
  int steps = 0;
  /* Ring AllReduce over 8 ranks: 14 steps, no scratch for fp32 */
  if (vc_plan_describe(VC_COLL_ALLREDUCE, VC_ALGO_RING, 8, 1 << 20, VC_FLOAT32, VC_SUM, 0, 0, 0, NULL, 0, &n,
                       &scratch, &steps) != VC_SUCCESS)
    return 3;
  if (steps != 14 || scratch != 0 || n == 0) return 4;
  vc_plan_entry_t* e = (vc_plan_entry_t*)malloc(n * sizeof(vc_plan_entry_t));
  if (vc_plan_describe(VC_COLL_ALLREDUCE, VC_ALGO_RING, 8, 1 << 20, VC_FLOAT32, VC_SUM, 0, 0, 0, e, n, &n,
                       &scratch, &steps) != VC_SUCCESS)
    return 5;
  if (e[0].step != 0 || e[0].reduce != 1) return 6;
  free(e);
  /* bad arguments are refused before any CUDA call */
  if (vc_allreduce(NULL, NULL, 8, 16, VC_FLOAT32, VC_SUM, VC_ALGO_RING, NULL) != VC_ERR_INVALID_ARG) return 7;
  vc_algo_t a;
  double t = 0;
  if (vc_select_algo(VC_COLL_ALLREDUCE, 8, 1 << 20, VC_FLOAT32, 0, &a, &t) != VC_SUCCESS || a != VC_ALGO_FUSED) return 8;
  /* execution-form settings: defaults, set, read back, restore */
  size_t v = 0;
  if (vc_get_copy_pipeline(&v) != VC_SUCCESS || v != VC_COPY_PIPELINE_DEFAULT) return 9;
  if (vc_set_copy_pipeline((size_t)-1) != VC_SUCCESS || vc_get_copy_pipeline(&v) != VC_SUCCESS || v != (size_t)-1)
    return 10;
  vc_set_copy_pipeline(VC_COPY_PIPELINE_DEFAULT);
  if (vc_get_single_launch(&v) != VC_SUCCESS || v != VC_SINGLE_LAUNCH_DEFAULT) return 11;
  if (vc_get_copy_pipeline(NULL) != VC_ERR_INVALID_ARG) return 12;
  if (vc_get_reuse_order(&v) != VC_SUCCESS || v != VC_REUSE_ORDER_DEFAULT) return 13;
  if (vc_set_reuse_order(0) != VC_SUCCESS || vc_get_reuse_order(&v) != VC_SUCCESS || v != 0) return 14;
  vc_set_reuse_order(VC_REUSE_ORDER_DEFAULT);
  if (vc_get_slice_limit(&v) != VC_SUCCESS || v != VC_SLICE_LIMIT_DEFAULT) return 15;
  if (vc_set_slice_limit(0) != VC_SUCCESS || vc_get_slice_limit(&v) != VC_SUCCESS || v != 0) return 16;
  vc_set_slice_limit(VC_SLICE_LIMIT_DEFAULT);
  {
    int m = 0;
    if (vc_get_merge_steps(&m) != VC_SUCCESS || m != 1) return 17;
    if (vc_set_merge_steps(0) != VC_SUCCESS || vc_get_merge_steps(&m) != VC_SUCCESS || m != 0) return 18;
    vc_set_merge_steps(1);
    if (vc_get_merge_steps(NULL) != VC_ERR_INVALID_ARG) return 19;
  }
  {
    /* 8 ranks, 1 MiB of fp32 per rank: the 14-step ring in one sliced launch;
       at 32 MiB per rank, above the slice limit, 14 launches */
    int form = -1, launches = -1, hr = -1;
    if (vc_plan_form(VC_COLL_ALLREDUCE, VC_ALGO_RING, 8, 1 << 18, VC_FLOAT32, VC_SUM, 0, 0, 0, &form, &launches,
                     &hr) != VC_SUCCESS || form != VC_FORM_SLICED || launches != 1 || hr != 0)
      return 20;
    if (vc_plan_form(VC_COLL_ALLREDUCE, VC_ALGO_RING, 8, (size_t)1 << 23, VC_FLOAT32, VC_SUM, 0, 0, 0, &form,
                     &launches, &hr) != VC_SUCCESS || form != VC_FORM_STEPS || launches != 14)
      return 21;
    if (vc_plan_form(VC_COLL_ALLREDUCE, VC_ALGO_RING, 8, 16, VC_FLOAT32, VC_SUM, 0, 0, 0, NULL, &launches, &hr) !=
        VC_ERR_INVALID_ARG)
      return 22;
  }
  printf("ok %d\n", vc_version());
  return 0;
}
