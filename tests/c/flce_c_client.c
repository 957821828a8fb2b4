/* A C99 client of include/flce.h: the header compiles as C, the library links, and calls
 * that need no device answer. Built and run by tests/test_abi_host.py on the CPU. */
#include <stdio.h>

#include "flce.h"

int main(void) {
  flce_options opt = {0};
  opt.weight_layout = FLCE_WEIGHT_VD;
  opt.input_dtype = FLCE_INPUT_BF16;
  /* N = 0 is refused by the argument checks, before any device is looked at */
  const flce_status st = flce_forward_ex((const void*)0, (const void*)0, (const int32_t*)0, 0, 128, 1024, -100,
                                         0.f, 0.f, FLCE_REDUCTION_MEAN, &opt, (float*)0, (float*)0, (void*)0, 0,
                                         (struct CUstream_st*)0);
  printf("%d %zu %d\n", flce_version(), flce_workspace_size(256, 128, 1024, 1), (int)st);
  printf("%s\n", flce_status_string(FLCE_ERR_F16_RANGE));
  return 0;
}
