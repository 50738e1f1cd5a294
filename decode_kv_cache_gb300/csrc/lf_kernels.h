// Internal table of compiled decode/prefill kernel instantiations.
#pragma once

#include <string>

namespace lf {

// Message returned by lf_last_error() on this thread.
void set_last_error(int code, const std::string& msg);  // message and status
// A call starts with no recorded failure (status LF_OK, empty message).
void clear_last_error();

enum KernelKind { kSimt = 0, kTensorCore = 1 };

struct KernelEntry {
  int kind = kSimt;               // kSimt: decode(DecodeArgs); kTensorCore: decode(TcArgs)
  const void* decode = nullptr;
  const void* decode_split = nullptr;  // kTensorCore: the split-launch instantiation
  const void* prefill = nullptr;  // __global__ void(PrefillArgs)
  const void* select = nullptr;   // __global__ void(DecodeArgs): layer-scope victim
  // Dynamic shared memory of one decode CTA; `items` bounds the units one
  // cluster visits per launch (tensor-core kernel only).
  int (*smem_bytes)(int stages, int chunk, int cluster, int evict, int items) = nullptr;
  int head_dim = 0, group = 0, elem_bytes = 0;
};

// Defined in one translation unit per element type.
bool find_kernels_bf16(int head_dim, int group, KernelEntry* out);
bool find_kernels_f32(int head_dim, int group, KernelEntry* out);
// tcgen05 path: bf16 storage, head_dim 128, group 1/2/4/8.
bool find_kernels_tc(int head_dim, int group, KernelEntry* out);

}  // namespace lf
