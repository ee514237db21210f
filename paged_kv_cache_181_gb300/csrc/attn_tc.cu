// tcgen05 (5th-generation tensor core) paged attention for bf16/f16 -- see below.
#include "common.cuh"

bool pkv_attn_tc_supports(pkv_dtype dt, int D) {
  (void)dt;
  (void)D;
  return false;
}

int pkv_launch_attn_tc(const PkvAttnArgs& a, pkv_dtype dt, void* stream) {
  (void)a;
  (void)dt;
  (void)stream;
  return -1;
}
