// diffattn_fwd_kv_noalloc: diffattn_fwd_kv on a fixed scratch area that the
// library owns, for callers that cannot provide a workspace.  Nothing is
// allocated: the scratch is a static device array of the module, and its
// address is looked up on every call (a context reset can move the module, so
// a cached address could go stale).
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = DIFFATTN_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes == (size_t{64} << 20), "64 MiB");

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch in the current device's context (nullptr on
// failure).  In host code g_scratch names a host-side stand-in, never the
// device array, so the kernels only ever receive this looked-up address.
void *scratch_address() {
  void *addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_scratch) != cudaSuccess) return nullptr;
  return addr;
}

}  // namespace

extern "C" {

diffattn_status diffattn_fwd_kv_noalloc(const diffattn_desc *desc, int64_t n_kv, const void *q1,
                                        const void *k1, const void *q2, const void *k2,
                                        const void *v, const float *lambda,
                                        const float *norm_w, void *out, int splits,
                                        void *stream) {
  int sp = 1;
  size_t need = 0;
  diffattn_status st = diffattn_fwd_kv_plan(desc, n_kv, splits, &sp, &need);
  if (st != DIFFATTN_OK) return st;
  if (need > kScratchBytes) return DIFFATTN_ERR_UNSUPPORTED;
  // The split-KV scratch holds no state that must start at zero (every block
  // that is read was written by the same call), so nothing is cleared.
  void *scratch = nullptr;
  if (need > 0 && (scratch = scratch_address()) == nullptr) return DIFFATTN_ERR_CUDA;
  return diffattn_fwd_kv(desc, n_kv, q1, k1, q2, k2, v, lambda, norm_w, out, sp, scratch,
                         need > 0 ? kScratchBytes : 0, stream);
}

}  // extern "C"
