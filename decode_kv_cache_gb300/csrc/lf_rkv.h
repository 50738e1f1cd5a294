// R-KV compression kernel: arguments and lookup (see lf_rkv.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace lf {

constexpr int kRkvMaxSlots = 4096;   // tokens of one unit a compression can hold

struct RkvArgs {
  CUtensorMap kmap;               // K slab as 2-D [rows][128] bf16, boxes {64, 64}
  const __nv_bfloat16* q_obs;     // [batch][alpha][q_heads][128] observation queries
  __nv_bfloat16* K;               // this layer's [batch][kv_heads][slot_stride][128]
  __nv_bfloat16* V;
  float* vnorm;                   // this layer's [batch][kv_heads][slot_stride]
  int32_t* pos;
  int32_t* count;                 // this layer's [batch][kv_heads]
  const int32_t* next_pos;
  int32_t* err;
  int kv_heads, q_heads, slot_stride, budget, alpha, beta, row_base;
  float lam, tau, scale_log2;     // lambda, cosine threshold, log2(e)/sqrt(128)
};

// Dynamic shared memory and threads of one compression CTA.
int rkv_smem_bytes();
int rkv_threads();
// __global__ void(RkvArgs) for q_heads / kv_heads = group, or null.
const void* find_rkv_kernel(int group);

}  // namespace lf
