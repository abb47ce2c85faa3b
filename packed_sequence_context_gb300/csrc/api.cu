// Host side of the C ABI declared in include/thd_attn.h: argument checks that
// need no device reads, workspace carving, TMA tensor maps, launches and the
// profiling hook.  The host never reads device memory and never synchronises.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "a2a.cuh"
#include "common.cuh"

namespace thd {

// ------------------------------------------------------------------ bookkeeping
static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 1;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

struct Prof {
  std::mutex mu;
  int kernel = 0;
  int max = 0;
  int n = 0;
  std::vector<cudaEvent_t> ev;
};
static Prof g_prof;

// One-shot test hook: the next launch of the armed kernel stalls on purpose
// (see thd_test_arm_stall).
static std::atomic<int> g_stall_kernel{0};
bool take_test_stall(int kernel_id) {
  int expect = kernel_id;
  return kernel_id != 0 && g_stall_kernel.compare_exchange_strong(expect, 0);
}

// Test hook: which forward kernel the next calls use (see
// thd_test_select_fwd_kernel); 0 = chosen from the workload.
static std::atomic<int> g_fwd_kernel{0};
int test_fwd_kernel() { return g_fwd_kernel.load(std::memory_order_relaxed); }

void prof_before(int id, cudaStream_t st) {
  if (g_prof.kernel != id) return;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (g_prof.kernel == id && g_prof.n < g_prof.max) cudaEventRecord(g_prof.ev[2 * g_prof.n], st);
}
void prof_after(int id, cudaStream_t st) {
  if (g_prof.kernel != id) return;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (g_prof.kernel == id && g_prof.n < g_prof.max) {
    cudaEventRecord(g_prof.ev[2 * g_prof.n + 1], st);
    ++g_prof.n;
  }
}

// ------------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over a [rows, H, D] bf16 THD tensor; box = 128 rows x 1 head x 64
// columns (128 bytes, the 128B-swizzle width).  Rows past the end read as 0.
static bool make_thd_map(CUtensorMap* m, const void* base, int64_t rows, int H, int D) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kTile};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

static int check_sizes(int B, int64_t T_q, int64_t T_kv, int Hq, int Hkv, int D, int cp, int pad_mode) {
  if (B < 1 || T_q < 0 || T_kv < 0 || Hq < 1 || Hkv < 1 || cp < 1 || cp > 1024) return THD_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return THD_ERR_INVALID_ARG;
  if (pad_mode < -1 || pad_mode > 1) return THD_ERR_INVALID_ARG;
  if (T_q >= (int64_t)1 << 31 || T_kv >= (int64_t)1 << 31 || B >= (1 << 24)) return THD_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return THD_ERR_UNSUPPORTED;
  return THD_OK;
}

static int check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (need == 0) return THD_ERR_INVALID_ARG;
  if (!ws || ws_bytes < need || !aligned(ws, 256)) return THD_ERR_WORKSPACE;
  return THD_OK;
}

static PlanParams plan_params(const int32_t* cu_q, const int32_t* cu_kv, const int32_t* pad_q,
                              const int32_t* pad_kv, int B, int cp, int causal, int pad_mode, int64_t rows_q,
                              int64_t rows_kv, int mode, char* ws, const WsLayout& L, int32_t* dev_status) {
  PlanParams p;
  std::memset(&p, 0, sizeof(p));
  p.cu_q = cu_q;
  p.cu_kv = cu_kv;
  p.pad_q = pad_q;
  p.pad_kv = pad_kv;
  p.B = B;
  p.cp = cp;
  p.causal = causal;
  p.pad_mode = pad_mode;
  p.rows_q = rows_q;
  p.rows_kv = rows_kv;
  p.mode = mode;
  p.step_lo = 0;
  p.step_hi = cp;
  p.eff = reinterpret_cast<int32_t*>(ws + L.eff);
  p.tile_off = reinterpret_cast<int32_t*>(ws + L.tile_off);
  p.counters = reinterpret_cast<int32_t*>(ws + L.counters);
  p.items = reinterpret_cast<int4*>(ws + L.items);
  p.item_cap = L.item_cap;
  p.dev_status = dev_status;
  return p;
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? THD_OK : THD_ERR_CUDA; }

// The merge keeps two weights per (head, token) of its tile in shared memory.
constexpr int kMergeMaxHeads = 16384;

// kv heads per locality group of the attention kernels' item order: the
// largest divisor of Hkv whose group re-reads at most kL2GroupBytes of
// operands (keys and values in the query-stationary kernels, queries and
// output gradients in the key-stationary one), so that while the group's
// items run those operands are read from HBM once and then hit in the
// 129 MB L2, leaving room for the streams that pass through once.
//
// The grouping pays only for long sequences: measured on GB300, it lifted
// the forward on one 131072-token sequence from 1166 to 1309 TFLOPS (DRAM
// reads per launch 12x lower), but on batches of short sequences (2-4K
// tokens) it made many CTAs read the same key tiles at once and lost 10-25%.
// So the order is grouped only when sequences average at least
// kLongSeqTokens rows; otherwise one group (entry-major, heads innermost).
constexpr size_t kL2GroupBytes = size_t(40) << 20;
constexpr int64_t kLongSeqTokens = 16384;
static bool long_sequences(int B, int64_t rows) { return rows >= kLongSeqTokens * (int64_t)B; }
static int locality_group(int Hkv, size_t bytes_per_kv_head, bool grouped) {
  if (!grouped) return Hkv;
  int best = 1;
  for (int d = 1; d <= Hkv; ++d)
    if (Hkv % d == 0 && (size_t)d * bytes_per_kv_head <= kL2GroupBytes) best = d;
  return best;
}

static int fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_q,
                      const int32_t* cu_kv, const int32_t* pad_q, const int32_t* pad_kv, int B, int64_t T_q,
                      int64_t T_kv, int Hq, int Hkv, int D, int causal, float scale, int cp, int pad_mode,
                      int step, bool part_fp32, void* ws, size_t ws_bytes, int32_t* dev_status, cudaStream_t st) {
  int rc = check_sizes(B, T_q, T_kv, Hq, Hkv, D, cp, pad_mode);
  if (rc) return rc;
  if (!q || !k || !v || !o || !lse || !cu_q || !cu_kv || !dev_status) return THD_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return THD_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale) || causal < kCausalNone || causal > kCausalBottomRight)
    return THD_ERR_INVALID_ARG;
  if (step >= cp) return THD_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(B, T_q, T_kv, Hq, D, cp, false);
  rc = check_ws(ws, ws_bytes, L.total);
  if (rc) return rc;
  char* w = static_cast<char*>(ws);
  PlanParams pp = plan_params(cu_q, cu_kv, pad_q, pad_kv, B, cp, causal, pad_mode, T_q, T_kv, 1, w, L, dev_status);
  if (step >= 0) {
    pp.step_lo = step;
    pp.step_hi = step + 1;
  }
  rc = cuda_status(launch_plan(pp, st));
  if (rc) return rc;
  CUtensorMap tk, tv;
  if (!make_thd_map(&tk, k, T_kv, Hkv, D) || !make_thd_map(&tv, v, T_kv, Hkv, D)) return THD_ERR_CUDA;
  FwdParams fp;
  std::memset(&fp, 0, sizeof(fp));
  fp.q = static_cast<const uint16_t*>(q);
  fp.o = o;
  fp.lse = lse;
  fp.eff = pp.eff;
  fp.items = pp.items;
  fp.counters = pp.counters;
  fp.claim = pp.counters + 1;
  // Sequences averaging >= kLongSeqTokens: the single-item kernel (three S
  // buffers keep the tensor pipe busy through the softmax), items grouped by
  // kv head and handed out dynamically.  Shorter sequences (items of a few
  // key tiles): the kernel with two items in flight per CTA, entry-major,
  // dynamic.  Measured on GB300: single-item 1311-1327 vs two-item 1093-1108
  // TFLOPS on one 131,072-token sequence; two-item 597 / 534 / 841 vs
  // single-item 519-535 / 515-521 / 835-848 on the 0.1-8K-token batches.
  const bool grouped = long_sequences(B, T_kv);
  fp.group_kv = locality_group(Hkv, (size_t)T_kv * D * 2 * 2, grouped);
  const int forced = test_fwd_kernel();
  const bool single = forced ? forced == THD_FWD_KERNEL_SINGLE : grouped;
  fp.dev_status = dev_status;
  fp.B = B;
  fp.Hq = Hq;
  fp.Hkv = Hkv;
  fp.cp = cp;
  fp.causal = causal;
  fp.T_q = T_q;
  fp.scale_log2 = scale * 1.4426950408889634f;
  fp.step_lo = pp.step_lo;
  fp.step_hi = pp.step_hi;
  fp.test_stall = take_test_stall(THD_KERNEL_FWD) ? 1 : 0;
  const int64_t bound = (int64_t)L.item_cap * Hq;
  const int grid = (int)(bound < num_sms() ? (bound > 0 ? bound : 1) : num_sms());
  // O is written in bf16 (the fused forward, or one step's partial in bf16)
  // or, for a step partial requested in fp32, in fp32
  const bool part32 = step >= 0 && part_fp32;
  return cuda_status(single ? launch_fwd(fp, tk, tv, D, part32, grouped, grid, st)
                            : launch_fwd_dual(fp, tk, tv, D, part32, grid, st));
}

// ------------------------------------------------------------------ A2A / hierarchical
// Sizes the emulated A2A layer accepts (see thd_cp_a2a in the header).
static int check_a2a_sizes(int B, int64_t T, int H, int D, int cp, int a2a) {
  if (B < 1 || B >= (1 << 24) || T < 0 || T >= ((int64_t)1 << 31) || H < 1 || D < 8 || D % 8 != 0)
    return THD_ERR_INVALID_ARG;
  if (cp < 1 || cp > 1024 || a2a < 1 || cp % a2a != 0 || H % a2a != 0 || T % cp != 0) return THD_ERR_INVALID_ARG;
  return THD_OK;
}

// Device-side checks of the padded offsets (the planner's validation alone):
// starts at 0, monotone, every P_b divisible by 2 cp, pad[B] <= T.  `cu` may
// be the valid-length offsets (also checked against the padded ones) or the
// padded offsets themselves.
static cudaError_t launch_a2a_checks(const int32_t* cu, const int32_t* pad, int B, int64_t T, int cp,
                                     int32_t* dev_status, cudaStream_t st) {
  PlanParams p;
  std::memset(&p, 0, sizeof(p));
  p.cu_q = cu;
  p.cu_kv = cu;
  p.pad_q = pad;
  p.pad_kv = pad;
  p.B = B;
  p.cp = cp;
  p.pad_mode = 1;
  p.rows_q = T;
  p.rows_kv = T;
  p.mode = 0;
  p.dev_status = dev_status;
  return launch_plan(p, st);
}

// The composites keep every member's buffer as a head slice of one tensor in
// global row order (the a2a_size = 1 layout of the move: member i's heads
// [i H/a2a, (i+1) H/a2a) side by side with the other members'), so ONE
// attention launch, with the P2P ring of cp/a2a ranks, serves all members; its
// work items are per head, so a member's outputs depend on its own slice only.
// Workspace: those global-order copies of the tensors, then the attention
// workspace.
struct A2aWs {
  size_t buf[8];  // q k v o (forward) + dO dQ dK dV (backward)
  size_t attn = 0;
  size_t total = 0;
};

static A2aWs a2a_ws_layout(int B, int64_t T, int Hq, int Hkv, int D, int cp, int a2a, bool bwd) {
  A2aWs w;
  size_t off = 0;
  const size_t bq = sizeof(uint16_t) * (size_t)T * Hq * D, bkv = sizeof(uint16_t) * (size_t)T * Hkv * D;
  const size_t sizes[8] = {bq, bkv, bkv, bq, bq, bq, bkv, bkv};
  const int n = bwd ? 8 : 4;
  for (int i = 0; i < 8; ++i) {
    w.buf[i] = off;
    if (i < n) off = align_up(off + sizes[i], 256);
  }
  w.attn = off;
  w.total = off + ws_layout(B, T, T, Hq, D, cp / a2a, bwd).total;
  return w;
}

static A2aJob a2a_job(const void* shard, void* groups, int H, int a2a) {
  A2aJob j;
  j.shard = const_cast<void*>(shard);
  j.groups = groups;
  j.Hg = H / a2a;
  return j;
}

static A2aParams a2a_params(const int32_t* pad, int B, int64_t T, int D, int cp, int a2a, const int32_t* dev_status) {
  A2aParams p;
  std::memset(&p, 0, sizeof(p));
  p.pad = pad;
  p.dev_status = dev_status;
  p.B = B;
  p.cp = cp;
  p.a2a = a2a;
  p.D = D;
  p.T = T;
  return p;
}

}  // namespace thd

using namespace thd;

extern "C" {

const char* thd_status_string(int s) {
  switch (s) {
    case THD_OK: return "ok";
    case THD_ERR_INVALID_ARG: return "invalid argument";
    case THD_ERR_UNSUPPORTED: return "unsupported configuration";
    case THD_ERR_CUDA: return "CUDA error";
    case THD_ERR_TIMEOUT: return "device wait timed out";
    case THD_ERR_WORKSPACE: return "workspace too small or misaligned";
    case THD_DEV_ERR_NONZERO_START: return "cu_seqlens must start at 0";
    case THD_DEV_ERR_NOT_MONOTONE: return "cu_seqlens not monotone";
    case THD_DEV_ERR_VALID_GT_PAD: return "valid length exceeds padded length";
    case THD_DEV_ERR_NOT_DIVISIBLE: return "padded length not divisible by 2*cp_size";
    case THD_DEV_ERR_EXCEEDS_BUF: return "sequences exceed the buffer rows";
    case THD_DEV_ERR_CAUSAL_LENGTHS: return "top-left causal attention needs equal q/kv lengths per sequence";
    case THD_DEV_ERR_CAPACITY: return "internal schedule capacity exceeded";
    default: return "unknown status";
  }
}

int thd_version(void) { return 100; }

size_t thd_workspace_size(int B, int64_t T_q, int64_t T_kv, int Hq, int Hkv, int D, int cp_size, int for_bwd) {
  if (check_sizes(B, T_q, T_kv, Hq, Hkv, D, cp_size, -1) != THD_OK) return 0;
  return ws_layout(B, T_q, T_kv, Hq, D, cp_size, for_bwd != 0).total;
}

int thd_cp_partition(const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded, int B, int cp_size,
                     int pad_between_seqs, int32_t* cu_rank, int32_t* cu_rank_padded, int32_t* cu_rank_half,
                     int32_t* token_map, int64_t token_map_capacity, int32_t* dev_status, thd_stream_t stream) {
  if (!cu_seqlens || !dev_status || B < 1 || cp_size < 1 || cp_size > 1024 || pad_between_seqs < -1 ||
      pad_between_seqs > 1)
    return THD_ERR_INVALID_ARG;
  if (token_map && token_map_capacity < 0) return THD_ERR_INVALID_ARG;
  PlanParams p;
  std::memset(&p, 0, sizeof(p));
  p.cu_q = cu_seqlens;
  p.cu_kv = cu_seqlens;
  p.pad_q = cu_seqlens_padded;
  p.pad_kv = cu_seqlens_padded;
  p.B = B;
  p.cp = cp_size;
  p.causal = 0;
  p.pad_mode = pad_between_seqs;
  p.rows_q = INT64_MAX;
  p.rows_kv = INT64_MAX;
  p.mode = 0;
  p.cu_rank = cu_rank;
  p.cu_rank_padded = cu_rank_padded;
  p.cu_rank_half = cu_rank_half;
  p.token_map = token_map;
  p.token_map_cap = token_map_capacity;
  p.dev_status = dev_status;
  return cuda_status(launch_plan(p, reinterpret_cast<cudaStream_t>(stream)));
}

int thd_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens_q,
                 const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                 const int32_t* cu_seqlens_kv_padded, int B, int64_t T_q, int64_t T_kv, int Hq, int Hkv, int D,
                 int causal, float softmax_scale, int cp_size, int pad_between_seqs, void* workspace,
                 size_t workspace_bytes, int32_t* dev_status, thd_stream_t stream) {
  return fwd_common(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded, B, T_q,
                    T_kv, Hq, Hkv, D, causal, softmax_scale, cp_size, pad_between_seqs, -1, false, workspace,
                    workspace_bytes, dev_status, reinterpret_cast<cudaStream_t>(stream));
}

int thd_attn_fwd_step(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                      const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                      const int32_t* cu_seqlens_kv_padded, int B, int64_t T_q, int64_t T_kv, int Hq, int Hkv,
                      int D, int causal, float softmax_scale, int cp_size, int pad_between_seqs, int step,
                      void* workspace, size_t workspace_bytes, int32_t* dev_status, thd_stream_t stream) {
  if (step < 0) return THD_ERR_INVALID_ARG;
  return fwd_common(q, k, v, o_part, lse_part, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                    cu_seqlens_kv_padded, B, T_q, T_kv, Hq, Hkv, D, causal, softmax_scale, cp_size,
                    pad_between_seqs, step, true, workspace, workspace_bytes, dev_status,
                    reinterpret_cast<cudaStream_t>(stream));
}

int thd_attn_fwd_step_bf16(const void* q, const void* k, const void* v, void* o_part, float* lse_part,
                           const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                           const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded, int B,
                           int64_t T_q, int64_t T_kv, int Hq, int Hkv, int D, int causal, float softmax_scale,
                           int cp_size, int pad_between_seqs, int step, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, thd_stream_t stream) {
  if (step < 0) return THD_ERR_INVALID_ARG;
  return fwd_common(q, k, v, o_part, lse_part, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                    cu_seqlens_kv_padded, B, T_q, T_kv, Hq, Hkv, D, causal, softmax_scale, cp_size,
                    pad_between_seqs, step, false, workspace, workspace_bytes, dev_status,
                    reinterpret_cast<cudaStream_t>(stream));
}

int thd_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int64_t dq_rows, int64_t dkv_rows, const int32_t* cu_seqlens_q,
                 const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                 const int32_t* cu_seqlens_kv_padded, int B, int64_t T_q, int64_t T_kv, int Hq, int Hkv, int D,
                 int causal, float softmax_scale, int cp_size, int pad_between_seqs, void* workspace,
                 size_t workspace_bytes, int32_t* dev_status, thd_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int rc = check_sizes(B, T_q, T_kv, Hq, Hkv, D, cp_size, pad_between_seqs);
  if (rc) return rc;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !cu_seqlens_q || !cu_seqlens_kv || !dev_status)
    return THD_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return THD_ERR_INVALID_ARG;
  if (dq_rows < T_q || dkv_rows < T_kv || dq_rows >= ((int64_t)1 << 31) || dkv_rows >= ((int64_t)1 << 31))
    return THD_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale) || causal < kCausalNone || causal > kCausalBottomRight)
    return THD_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(B, T_q, T_kv, Hq, D, cp_size, true);
  rc = check_ws(workspace, workspace_bytes, L.total);
  if (rc) return rc;
  char* w = static_cast<char*>(workspace);
  // one planner launch, two schedules: key tiles for the dK/dV pass, query
  // tiles for the dQ pass
  PlanParams pp = plan_params(cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded, B, cp_size,
                              causal, pad_between_seqs, T_q, T_kv, 3, w, L, dev_status);
  pp.tile_off_q = reinterpret_cast<int32_t*>(w + L.tile_off_q);
  pp.counters_q = reinterpret_cast<int32_t*>(w + L.counters_q);
  pp.items_q = reinterpret_cast<int4*>(w + L.items_q);
  pp.item_cap_q = L.item_cap_q;
  rc = cuda_status(launch_plan(pp, st));
  if (rc) return rc;
  float* delta = reinterpret_cast<float*>(w + L.delta);
  float* lse2 = reinterpret_cast<float*>(w + L.lse2);
  rc = cuda_status(launch_bwd_prep(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), lse, delta,
                                   lse2, pp.eff, B, T_q, Hq, D, dev_status, st));
  if (rc) return rc;
  CUtensorMap tq, tdo, tk, tv;
  if (!make_thd_map(&tq, q, T_q, Hq, D) || !make_thd_map(&tdo, dout, T_q, Hq, D) ||
      !make_thd_map(&tk, k, T_kv, Hkv, D) || !make_thd_map(&tv, v, T_kv, Hkv, D))
    return THD_ERR_CUDA;
  DqParams dp;
  std::memset(&dp, 0, sizeof(dp));
  dp.q = static_cast<const uint16_t*>(q);
  dp.dout = static_cast<const uint16_t*>(dout);
  dp.lse2 = lse2;
  dp.delta = delta;
  dp.dq = static_cast<uint16_t*>(dq);
  dp.eff = pp.eff;
  dp.items = pp.items_q;
  dp.counters = pp.counters_q;
  dp.claim = pp.counters_q + 1;
  const bool grouped_q = long_sequences(B, T_kv);
  dp.group_kv = locality_group(Hkv, (size_t)T_kv * D * 2 * 2, grouped_q);
  dp.dev_status = dev_status;
  dp.B = B;
  dp.Hq = Hq;
  dp.Hkv = Hkv;
  dp.cp = cp_size;
  dp.causal = causal;
  dp.T_q = T_q;
  dp.dq_rows = dq_rows;
  dp.scale = softmax_scale;
  dp.scale_log2 = softmax_scale * 1.4426950408889634f;
  dp.step_lo = 0;
  dp.step_hi = cp_size;
  dp.test_stall = take_test_stall(THD_KERNEL_BWD_DQ) ? 1 : 0;
  const int64_t bound_q = (int64_t)L.item_cap_q * Hq;
  const int grid_q = (int)(bound_q < num_sms() ? (bound_q > 0 ? bound_q : 1) : num_sms());
  rc = cuda_status(launch_dq(dp, tk, tv, D, grouped_q, grid_q, st));
  if (rc) return rc;
  BwdParams bp;
  std::memset(&bp, 0, sizeof(bp));
  bp.q = static_cast<const uint16_t*>(q);
  bp.dout = static_cast<const uint16_t*>(dout);
  bp.lse2 = lse2;
  bp.delta = delta;
  bp.dk = static_cast<uint16_t*>(dk);
  bp.dv = static_cast<uint16_t*>(dv);
  bp.eff = pp.eff;
  bp.items = pp.items;
  bp.counters = pp.counters;
  bp.claim = pp.counters + 1;
  const bool grouped_kv = long_sequences(B, T_q);
  bp.group_kv = locality_group(Hkv, (size_t)T_q * (Hq / Hkv) * (D * 2 * 2 + 8), grouped_kv);
  bp.dev_status = dev_status;
  bp.B = B;
  bp.Hq = Hq;
  bp.Hkv = Hkv;
  bp.cp = cp_size;
  bp.causal = causal;
  bp.T_q = T_q;
  bp.dkv_rows = dkv_rows;
  bp.scale = softmax_scale;
  bp.scale_log2 = softmax_scale * 1.4426950408889634f;
  bp.test_stall = take_test_stall(THD_KERNEL_BWD) ? 1 : 0;
  const int64_t bound = (int64_t)L.item_cap * Hkv;
  const int grid = (int)(bound < num_sms() ? (bound > 0 ? bound : 1) : num_sms());
  return cuda_status(launch_bwd(bp, tq, tdo, tk, tv, D, grouped_kv, grid, st));
}

int thd_lse_merge(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part, int64_t T, int H, int D,
                  thd_stream_t stream) {
  if (!o_acc || !lse_acc || !o_part || !lse_part || T < 0 || H < 1 || D < 4 || D % 4 != 0) return THD_ERR_INVALID_ARG;
  if (!aligned(o_acc, 16) || !aligned(o_part, 16)) return THD_ERR_INVALID_ARG;
  if (H > kMergeMaxHeads) return THD_ERR_UNSUPPORTED;
  return cuda_status(launch_lse_merge(o_acc, lse_acc, o_part, lse_part, T, H, D, reinterpret_cast<cudaStream_t>(stream)));
}

int thd_lse_merge_bf16(float* o_acc, float* lse_acc, const void* o_part, const float* lse_part, int64_t T, int H,
                       int D, thd_stream_t stream) {
  if (!o_acc || !lse_acc || !o_part || !lse_part || T < 0 || H < 1 || D < 4 || D % 4 != 0) return THD_ERR_INVALID_ARG;
  if (!aligned(o_acc, 16) || !aligned(o_part, 8)) return THD_ERR_INVALID_ARG;
  if (H > kMergeMaxHeads) return THD_ERR_UNSUPPORTED;
  return cuda_status(launch_lse_merge_bf16(o_acc, lse_acc, static_cast<const uint16_t*>(o_part), lse_part, T, H, D,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

int thd_grad_tail_zero(void* dq, void* dk, void* dv, int64_t dq_rows, int64_t dkv_rows, int Hq, int Hkv, int D,
                       const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded, int B,
                       int host_knows_no_tail, thd_stream_t stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || D < 8 || D % 8 != 0 || dq_rows < 0 || dkv_rows < 0) return THD_ERR_INVALID_ARG;
  if (dq && !cu_seqlens_q_padded) return THD_ERR_INVALID_ARG;
  if ((dk || dv) && !cu_seqlens_kv_padded) return THD_ERR_INVALID_ARG;
  if (!aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16)) return THD_ERR_INVALID_ARG;
  if (host_knows_no_tail) return THD_OK;  // nothing to clear: no launch at all
  if (!dq && !dk && !dv) return THD_OK;
  return cuda_status(launch_tail_zero(static_cast<uint16_t*>(dq), static_cast<uint16_t*>(dk),
                                      static_cast<uint16_t*>(dv), dq_rows, dkv_rows, Hq, Hkv, D,
                                      cu_seqlens_q_padded ? cu_seqlens_q_padded + B : nullptr,
                                      cu_seqlens_kv_padded ? cu_seqlens_kv_padded + B : nullptr, nullptr,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

int thd_cp_a2a(const void* src, void* dst, const int32_t* cu_seqlens_padded, int B, int64_t T, int H, int D,
               int cp_size, int a2a_size, int direction, int32_t* dev_status, thd_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int rc = check_a2a_sizes(B, T, H, D, cp_size, a2a_size);
  if (rc) return rc;
  if (!src || !dst || !cu_seqlens_padded || !dev_status || !aligned(src, 16) || !aligned(dst, 16))
    return THD_ERR_INVALID_ARG;
  if (direction != THD_A2A_TO_GROUPS && direction != THD_A2A_TO_SHARDS) return THD_ERR_INVALID_ARG;
  rc = cuda_status(launch_a2a_checks(cu_seqlens_padded, cu_seqlens_padded, B, T, cp_size, dev_status, st));
  if (rc) return rc;
  A2aParams p = a2a_params(cu_seqlens_padded, B, T, D, cp_size, a2a_size, dev_status);
  const bool to_groups = direction == THD_A2A_TO_GROUPS;
  p.job[0] = to_groups ? a2a_job(src, dst, H, a2a_size) : a2a_job(dst, const_cast<void*>(src), H, a2a_size);
  p.njobs = 1;
  return cuda_status(launch_a2a(p, to_groups, st));
}

size_t thd_a2a_workspace_size(int B, int64_t T, int Hq, int Hkv, int D, int cp_size, int a2a_size, int for_bwd) {
  if (check_a2a_sizes(B, T, Hq, D, cp_size, a2a_size) != THD_OK || Hkv < 1 || Hkv % a2a_size != 0) return 0;
  if (check_sizes(B, T, T, Hq, Hkv, D, cp_size / a2a_size, -1) != THD_OK) return 0;
  return a2a_ws_layout(B, T, Hq, Hkv, D, cp_size, a2a_size, for_bwd != 0).total;
}

// Shared checks of the two composites; returns the layout through `L`.
static int a2a_composite_checks(const int32_t* cu, const int32_t* pad, int B, int64_t T, int Hq, int Hkv, int D,
                                int causal, float scale, int cp, int a2a, void* ws, size_t ws_bytes,
                                const int32_t* dev_status, bool bwd, A2aWs& L) {
  int rc = check_a2a_sizes(B, T, Hq, D, cp, a2a);
  if (rc) return rc;
  if (Hkv < 1 || Hkv % a2a != 0) return THD_ERR_INVALID_ARG;
  rc = check_sizes(B, T, T, Hq, Hkv, D, cp / a2a, -1);
  if (rc) return rc;
  if (!cu || !pad || !dev_status) return THD_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale) || (causal != 0 && causal != 1)) return THD_ERR_INVALID_ARG;
  L = a2a_ws_layout(B, T, Hq, Hkv, D, cp, a2a, bwd);
  return check_ws(ws, ws_bytes, L.total);
}

int thd_attn_fwd_a2a(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens,
                     const int32_t* cu_seqlens_padded, int B, int64_t T, int Hq, int Hkv, int D, int causal,
                     float softmax_scale, int cp_size, int a2a_size, void* workspace, size_t workspace_bytes,
                     int32_t* dev_status, thd_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  A2aWs L;
  int rc = a2a_composite_checks(cu_seqlens, cu_seqlens_padded, B, T, Hq, Hkv, D, causal, softmax_scale, cp_size,
                                a2a_size, workspace, workspace_bytes, dev_status, false, L);
  if (rc) return rc;
  if (!q || !k || !v || !o || !lse || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return THD_ERR_INVALID_ARG;
  char* w = static_cast<char*>(workspace);
  const int p2p = cp_size / a2a_size;
  rc = cuda_status(launch_a2a_checks(cu_seqlens, cu_seqlens_padded, B, T, cp_size, dev_status, st));
  if (rc) return rc;
  A2aParams in = a2a_params(cu_seqlens_padded, B, T, D, cp_size, 1, dev_status);
  in.job[0] = a2a_job(q, w + L.buf[0], Hq, 1);
  in.job[1] = a2a_job(k, w + L.buf[1], Hkv, 1);
  in.job[2] = a2a_job(v, w + L.buf[2], Hkv, 1);
  in.njobs = 3;
  rc = cuda_status(launch_a2a(in, true, st));
  if (rc) return rc;
  rc = fwd_common(w + L.buf[0], w + L.buf[1], w + L.buf[2], w + L.buf[3], lse, cu_seqlens, cu_seqlens,
                  cu_seqlens_padded, cu_seqlens_padded, B, T, T, Hq, Hkv, D, causal, softmax_scale, p2p, -1, -1,
                  false, w + L.attn, workspace_bytes - L.attn, dev_status, st);
  if (rc) return rc;
  A2aParams out = a2a_params(cu_seqlens_padded, B, T, D, cp_size, 1, dev_status);
  out.job[0] = a2a_job(o, w + L.buf[3], Hq, 1);
  out.njobs = 1;
  return cuda_status(launch_a2a(out, false, st));
}

int thd_attn_bwd_a2a(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded, int B,
                     int64_t T, int Hq, int Hkv, int D, int causal, float softmax_scale, int cp_size, int a2a_size,
                     void* workspace, size_t workspace_bytes, int32_t* dev_status, thd_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  A2aWs L;
  int rc = a2a_composite_checks(cu_seqlens, cu_seqlens_padded, B, T, Hq, Hkv, D, causal, softmax_scale, cp_size,
                                a2a_size, workspace, workspace_bytes, dev_status, true, L);
  if (rc) return rc;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return THD_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return THD_ERR_INVALID_ARG;
  char* w = static_cast<char*>(workspace);
  const int p2p = cp_size / a2a_size;
  rc = cuda_status(launch_a2a_checks(cu_seqlens, cu_seqlens_padded, B, T, cp_size, dev_status, st));
  if (rc) return rc;
  A2aParams in = a2a_params(cu_seqlens_padded, B, T, D, cp_size, 1, dev_status);
  in.job[0] = a2a_job(q, w + L.buf[0], Hq, 1);
  in.job[1] = a2a_job(k, w + L.buf[1], Hkv, 1);
  in.job[2] = a2a_job(v, w + L.buf[2], Hkv, 1);
  in.job[3] = a2a_job(o, w + L.buf[3], Hq, 1);
  in.job[4] = a2a_job(dout, w + L.buf[4], Hq, 1);
  in.njobs = 5;
  rc = cuda_status(launch_a2a(in, true, st));
  if (rc) return rc;
  rc = thd_attn_bwd(w + L.buf[0], w + L.buf[1], w + L.buf[2], w + L.buf[3], lse, w + L.buf[4], w + L.buf[5],
                    w + L.buf[6], w + L.buf[7], T, T, cu_seqlens, cu_seqlens, cu_seqlens_padded, cu_seqlens_padded,
                    B, T, T, Hq, Hkv, D, causal, softmax_scale, p2p, -1, w + L.attn, workspace_bytes - L.attn,
                    dev_status, stream);
  if (rc) return rc;
  A2aParams out = a2a_params(cu_seqlens_padded, B, T, D, cp_size, 1, dev_status);
  out.job[0] = a2a_job(dq, w + L.buf[5], Hq, 1);
  out.job[1] = a2a_job(dk, w + L.buf[6], Hkv, 1);
  out.job[2] = a2a_job(dv, w + L.buf[7], Hkv, 1);
  out.njobs = 3;
  return cuda_status(launch_a2a(out, false, st));
}

int thd_profile_enable(int kernel_id, int max_records) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  for (auto e : g_prof.ev) cudaEventDestroy(e);
  g_prof.ev.clear();
  g_prof.kernel = 0;
  g_prof.n = 0;
  g_prof.max = 0;
  if (kernel_id == 0 || max_records <= 0) return THD_OK;
  g_prof.ev.resize(2 * (size_t)max_records);
  for (auto& e : g_prof.ev)
    if (cudaEventCreate(&e) != cudaSuccess) return THD_ERR_CUDA;
  g_prof.max = max_records;
  g_prof.kernel = kernel_id;
  return THD_OK;
}

int thd_profile_read(float* ms_out, int max_out, int* count_out) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  const int n = g_prof.n < max_out ? g_prof.n : max_out;
  for (int i = 0; i < n; ++i) {
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess) return THD_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess) return THD_ERR_CUDA;
    if (ms_out) ms_out[i] = ms;
  }
  if (count_out) *count_out = n;
  return THD_OK;
}

uint64_t thd_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int thd_test_select_fwd_kernel(int which) {
  if (which != 0 && which != THD_FWD_KERNEL_SINGLE && which != THD_FWD_KERNEL_DUAL) return THD_ERR_INVALID_ARG;
  g_fwd_kernel.store(which, std::memory_order_relaxed);
  return THD_OK;
}

int thd_test_arm_stall(int kernel_id) {
  if (kernel_id != 0 && kernel_id != THD_KERNEL_FWD && kernel_id != THD_KERNEL_BWD && kernel_id != THD_KERNEL_BWD_DQ)
    return THD_ERR_INVALID_ARG;
  g_stall_kernel.store(kernel_id);
  return THD_OK;
}

}  // extern "C"
