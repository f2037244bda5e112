#include "internal.h"
spear_status_t spear_launch_prefill(spear_linear_s*, const __nv_bfloat16*, __nv_bfloat16*, int, cudaStream_t) {
  return SPEAR_ERR_UNSUPPORTED;
}
