// thd_attn_fwd_noalloc: the forward pass for callers that cannot allocate
// device memory where they call it.  Its scratch (the effective metadata,
// tile offsets and longest-first schedule that thd_attn_fwd keeps in the
// caller's workspace) lives in the file-scope device array below instead.
#include <mutex>

#include "common.cuh"

namespace {

// Every GPU that loads this library holds this array until the process exits.
__device__ __align__(256) uint8_t g_fwd_scratch[THD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_fwd_scratch on the current device, looked up once per
// device.  In host code `g_fwd_scratch` names a host-side stand-in, never the
// device array, so it must not be handed to a kernel directly.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return THD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return THD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || !p) return THD_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return THD_OK;
}

}  // namespace

extern "C" int thd_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                                    const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded, int B,
                                    int64_t T_q, int64_t T_kv, int Hq, int Hkv, int D, int causal,
                                    float softmax_scale, int cp_size, int pad_between_seqs, int32_t* dev_status,
                                    thd_stream_t stream) {
  const size_t need = thd_workspace_size(B, T_q, T_kv, Hq, Hkv, D, cp_size, 0);
  // sizes thd_attn_fwd rejects: let it report them (same code, nothing launched)
  if (need == 0)
    return thd_attn_fwd(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded, B,
                        T_q, T_kv, Hq, Hkv, D, causal, softmax_scale, cp_size, pad_between_seqs, nullptr, 0,
                        dev_status, stream);
  if (need > (size_t)THD_NOALLOC_SCRATCH_BYTES) return THD_ERR_WORKSPACE;  // beyond the static maximum
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != THD_OK) return rc;
  // Nothing in the scratch has to start at zero: the planner kernel of this
  // call writes everything the forward kernel reads.
  return thd_attn_fwd(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded, B,
                      T_q, T_kv, Hq, Hkv, D, causal, softmax_scale, cp_size, pad_between_seqs, scratch,
                      (size_t)THD_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
