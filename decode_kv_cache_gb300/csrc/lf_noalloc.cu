// lf_prefill_fill_noalloc: the prefill step for callers that cannot allocate
// device memory (see include/longflow.h).
//
// The prefill kernel reads each sequence's prompt length from device memory.
// lf_prefill_fill keeps those lengths in memory that lf_cache_create_ex
// allocated; this entry point instead uses a fixed array compiled into the
// library, so a caller that owns the slab memory itself can run the prefill
// without any allocation.  The array is shared by every call on a device and
// keeps the last call's contents (the call overwrites the first `batch`
// entries before the kernel reads them); calls whose kernels overlap on the
// GPU race on it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "lf_decode.cuh"
#include "lf_kernels.h"
#include "longflow.h"

namespace {

constexpr int kMaxDevices = 64;

// One prompt length per sequence: 64 KB on every device that loads the library.
__device__ __align__(256) int32_t g_prompt_len_scratch[LF_NOALLOC_MAX_BATCH];

std::mutex g_setup_mutex;
// Per device: the array's address and the id of the CUDA context it was
// looked up in.  A cudaDeviceReset in the process ends that context (the next
// runtime call makes a new one, where the array may sit elsewhere), so the
// address is looked up again whenever the current context's id differs.
int32_t* g_scratch_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

int noalloc_fail(int code, const std::string& msg) {
  lf::set_last_error(code, msg);
  return code;
}

// Id of the current CUDA context (unique over the process's lifetime), or 0
// if the driver does not tell.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {  // called with g_setup_mutex held
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(fn);
    (void)cudaGetLastError();
    looked_up = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch array on the current device: looked up once
// per device (and again after the device's context was replaced), with that
// device current.
int scratch_address(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return noalloc_fail(LF_ERR_CUDA, cudaGetErrorString(e));
  }
  if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(LF_ERR_ARG, "device index too large");
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev] || current_context_id() != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_prompt_len_scratch);
    if (e != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return noalloc_fail(LF_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    }
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    // read after the lookup, which makes the device's context current if the
    // runtime had not yet
    g_scratch_ctx[dev] = current_context_id();
  }
  *out = g_scratch_ptr[dev];
  return LF_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int lf_prefill_fill_noalloc(const lf_layout* dst, int layer, const void* k,
                                       const void* v, const int32_t* prompt_len, int max_prompt,
                                       lf_stream_t stream) {
  lf::clear_last_error();
  if (!dst) return noalloc_fail(LF_ERR_ARG, "null destination layout");
  if (!dst->k || !dst->v || !dst->vnorm || !dst->pos || !dst->count || !dst->next_pos)
    return noalloc_fail(LF_ERR_ARG, "destination layout has a null pointer");
  if (layer < 0 || layer >= dst->layers) return noalloc_fail(LF_ERR_ARG, "layer out of range");
  if (dst->norm != 0 && dst->norm != 1 && dst->norm != 2)
    return noalloc_fail(LF_ERR_ARG, "norm must be 0 (l1), 1 or 2");
  if (dst->batch < 1 || dst->kv_heads < 1 || dst->capacity < 1 ||
      dst->slot_stride < dst->capacity || dst->slot_stride % 4 != 0)
    return noalloc_fail(LF_ERR_ARG, "invalid destination shape");
  if (dst->batch > LF_NOALLOC_MAX_BATCH)
    return noalloc_fail(LF_ERR_ARG, "batch " + std::to_string(dst->batch) +
                                        " exceeds LF_NOALLOC_MAX_BATCH (" +
                                        std::to_string(LF_NOALLOC_MAX_BATCH) + ")");
  if (!prompt_len || max_prompt < 0) return noalloc_fail(LF_ERR_ARG, "bad prompt lengths");
  // Deferred mode (a pending array): the step that fills the buffer chooses
  // the first victim, so a prompt leaves at least one slot free.
  const int limit = dst->pending ? dst->capacity - 1 : dst->capacity;
  int longest = 0;
  for (int b = 0; b < dst->batch; ++b) {
    const int P = prompt_len[b];
    if (P < 0 || P > max_prompt || P > limit)
      return noalloc_fail(LF_ERR_ARG, "prompt_len[" + std::to_string(b) + "] = " +
                                          std::to_string(P) + " outside [0, min(max_prompt, " +
                                          (dst->pending ? "capacity - 1 (deferred mode))]"
                                                        : "capacity)]"));
    if (P > longest) longest = P;
  }
  if (longest > 0 && (!k || !v || !aligned16(k) || !aligned16(v)))
    return noalloc_fail(LF_ERR_ARG, "k and v must be non-null and 16-byte aligned");
  if (!aligned16(dst->k) || !aligned16(dst->v))
    return noalloc_fail(LF_ERR_ARG, "destination K and V must be 16-byte aligned");
  lf::KernelEntry kern;
  const bool found = (dst->dtype == LF_BF16) ? lf::find_kernels_bf16(dst->head_dim, 1, &kern)
                     : (dst->dtype == LF_F32) ? lf::find_kernels_f32(dst->head_dim, 1, &kern)
                                              : false;
  if (!found) return noalloc_fail(LF_ERR_UNSUPPORTED, "unsupported dtype or head_dim");

  int32_t* plen = nullptr;
  int rc = scratch_address(&plen);
  if (rc != LF_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(plen, prompt_len, (size_t)dst->batch * 4,
                                  cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return noalloc_fail(LF_ERR_CUDA, std::string("uploading prompt lengths: ") + cudaGetErrorString(e));
  }
  const size_t layer_units = (size_t)dst->batch * dst->kv_heads;
  const size_t layer_slots = layer_units * dst->slot_stride;
  const size_t elem = (size_t)kern.elem_bytes;
  lf::PrefillArgs a;
  a.k = k;
  a.v = v;
  a.plen = plen;
  a.K = static_cast<char*>(dst->k) + layer * layer_slots * dst->head_dim * elem;
  a.V = static_cast<char*>(dst->v) + layer * layer_slots * dst->head_dim * elem;
  a.vnorm = dst->vnorm + layer * layer_slots;
  a.pos = dst->pos + layer * layer_slots;
  a.count = dst->count + layer * layer_units;
  a.next_pos = dst->next_pos + layer * layer_units;
  a.acc = dst->acc ? dst->acc + layer * layer_slots : nullptr;
  a.pending = dst->pending ? dst->pending + layer * layer_units : nullptr;
  a.kv_heads = dst->kv_heads;
  a.max_prompt = max_prompt;
  a.slot_stride = dst->slot_stride;
  a.norm = (dst->norm == 2) ? 2 : 1;
  void* args[] = {&a};
  e = cudaLaunchKernel(kern.prefill, dim3(dst->kv_heads, dst->batch, 1), dim3(lf::kThreads, 1, 1),
                       args, 0, st);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return noalloc_fail(LF_ERR_CUDA, std::string("prefill launch: ") + cudaGetErrorString(e));
  }
  return LF_OK;
}
