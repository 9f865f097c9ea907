// C ABI of the B300 DeepSeekMoE layer (declarations and contracts: moe.h).
//
// Host side only marshals: it validates arguments, lays out the workspace,
// encodes TMA tensor maps and enqueues kernels on the caller's stream.  It
// never allocates device memory, never synchronises (except
// moe_read_device_status, whose job that is) and never reads device data.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "expert_gemm.cuh"
#include "fp8_gemm.cuh"
#include "backward.cuh"
#include "kernels.cuh"
#include "moe.h"
#include "wgrad_gemm.cuh"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// E4M3 expert GEMMs, with amax/448 scales or with UE8M0 (power-of-two) scales.
bool is_fp8(const moe_dims& d) { return d.prec == MOE_FP8_E4M3 || d.prec == MOE_FP8_UE8M0; }

// Entries of the chunk -> group table: at most rows/128 + one partial chunk
// per group (chunks are >= 128 rows).
int64_t cgroup_cap(const moe_dims& d) {
  return (int64_t(d.T) * d.k + 127) / 128 + d.E + d.n_shared + 1;
}

// K splits of the router logits GEMM: more CTAs for the centroid stream when
// there are few tokens (up to the 148 SMs of a B300, at most 8 splits), at
// most 2^21 fp32 partial logits in all (the scratch of moe_route_noalloc
// holds that many).
struct LogitsSplit {
  int splits, kb_per_split;
};

LogitsSplit logits_split(const moe_dims& d) {
  const int64_t tiles = ((int64_t(d.T) + 127) / 128) * ((int64_t(d.E) + 127) / 128);
  const int num_kb = (d.d + 63) / 64;
  // at most 8 splits: the top-k kernel reads every split's partial logits
  // (16 made the decode step's router no faster and its top-k slower)
  int64_t want = tiles > 0 ? 148 / tiles : 1;
  if (want > 8) want = 8;
  const int64_t te = int64_t(d.T) * d.E;
  if (te > 0 && want * te > MOE_ROUTE_NOALLOC_MAX_LOGITS) want = MOE_ROUTE_NOALLOC_MAX_LOGITS / te;
  if (want < 1) want = 1;
  if (want > num_kb) want = num_kb;
  const int kb_per = static_cast<int>((num_kb + want - 1) / want);
  return LogitsSplit{(num_kb + kb_per - 1) / kb_per, kb_per};
}

// Byte offsets of every buffer inside the caller's workspace.
struct Layout {
  size_t status, queue, z, idx, gate, counts, mask, wprefix, cnt, offsets, groups, mt_total, cgroup, perm, slot;
  size_t x, xs, uq, uqs, h, hs, hsh, hshs, y, ysh, total;
};

Layout make_layout(const moe_dims& d) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes > 0 ? bytes : 1);
    return o;
  };
  const int64_t T = d.T, R = T * d.k, W = (T + 31) / 32, E = d.E, I = d.inter, D = d.d, Ns = d.n_shared;
  const bool fp8 = is_fp8(d);
  const int64_t eb = fp8 ? 1 : 2;  // bytes per GEMM operand element
  L.status = take(256);
  L.queue = take(4 * sizeof(int));  // item counters of the four expert GEMM launches
  L.z = take(logits_split(d).splits * T * E * 4);
  L.idx = take(R * 4);
  L.gate = take(R * 4);
  L.counts = take(E * 4);
  L.mask = take(E * W * 4);
  L.wprefix = take(E * W * 4);
  L.cnt = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.groups = take((E + Ns + 1) * sizeof(GroupEntry));
  L.mt_total = take(16);
  L.cgroup = take(cgroup_cap(d) * 4);
  L.perm = take(R * 4);
  L.slot = take(R * 4);
  L.x = take(R * D * eb);
  L.xs = fp8 ? take(D / 128 * R * 4) : 0;
  L.uq = fp8 ? take(T * D) : 0;
  L.uqs = fp8 ? take(D / 128 * T * 4) : 0;
  L.h = take(R * I * eb);
  L.hs = fp8 ? take(I / 128 * R * 4) : 0;
  L.hsh = take(Ns * T * I * eb);
  L.hshs = fp8 ? take(I / 128 * Ns * T * 4) : 0;
  L.y = take(R * D * 2);
  L.ysh = take(Ns * T * D * 2);
  L.total = off;
  return L;
}

template <class P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool d_T_nonzero(const moe_dims* d) { return d->T != 0; }

moe_status check_dims(const moe_dims* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->d <= 0 || d->E <= 0 || d->k <= 0 || d->n_shared < 0 || d->inter <= 0) return MOE_ERR_INVALID_ARG;
  if (d->prec != MOE_BF16 && d->prec != MOE_FP8_E4M3 && d->prec != MOE_FP8_UE8M0) return MOE_ERR_INVALID_ARG;
  if (d->k > d->E || d->k > 32) return MOE_ERR_INVALID_ARG;
  if (d->E > 1024) return MOE_ERR_UNSUPPORTED;
  if (d->d % 128 != 0 || d->inter % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->T) * d->k > (int64_t(1) << 30)) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->n_shared) * d->T > (int64_t(1) << 30)) return MOE_ERR_UNSUPPORTED;
  if (d->route_groups < 0 || d->route_group_limit < 0) return MOE_ERR_INVALID_ARG;
  if (d->route_groups > 0) {
    if (d->route_groups > 32) return MOE_ERR_UNSUPPORTED;
    if (d->E % d->route_groups != 0 || d->route_group_limit < 1 || d->route_group_limit > d->route_groups ||
        int64_t(d->route_group_limit) * (d->E / d->route_groups) < d->k)
      return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

moe_status check_ws(const moe_dims* d, const void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < make_layout(*d).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status cuda_ok(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }
moe_status launched() { return cuda_ok(cudaGetLastError()); }

#define MOE_TRY(expr)                       \
  do {                                      \
    const moe_status _s = (expr);           \
    if (_s != MOE_OK) return _s;            \
  } while (0)

// Optional stage timing: records caller-created CUDA events between stages.
struct Recorder {
  void* const* ev = nullptr;
  int n = 0, i = 0;
  cudaStream_t st = nullptr;
  moe_status mark() {
    if (!ev) return MOE_OK;
    if (i >= n) return MOE_ERR_INVALID_ARG;
    return cuda_ok(cudaEventRecord(static_cast<cudaEvent_t>(ev[i++]), st));
  }
};

// ------------------------------------------------------------------ TMA maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 2-D K-major operand [rows, K]: boxes of 128 bytes of K by box_rows rows,
// 128-byte swizzle, zero fill outside the tensor.
moe_status make_tmap(CUtensorMap* map, const void* base, bool fp8, int64_t rows, int64_t K, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * (fp8 ? 1 : 2))};
  const cuuint32_t box[2] = {fp8 ? 128u : 64u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

GemmArgs base_args(int* status) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.status = status;
  return a;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Token rows per chunk of the expert GEMMs (the N of one MMA at most).
constexpr int kChunkBf16 = kXChunk;
constexpr int kChunkFp8 = 128;
int chunk_rows(const moe_dims& d) { return is_fp8(d) ? kChunkFp8 : kChunkBf16; }

// ------------------------------------------------------------------ pieces
// Router logits (tcgen05 GEMM, bf16 in, fp32 out) then the warp-per-token top-k.
moe_status enqueue_route(const moe_dims& d, const uint16_t* u, const uint16_t* cent, const float* bias, int32_t* idx,
                         float* gate, int32_t* counts, uint32_t* mask, float* z, int* status, cudaStream_t st,
                         Recorder* rec = nullptr) {
  const int W = (d.T + 31) / 32;
  MOE_TRY(cuda_ok(cudaMemsetAsync(counts, 0, sizeof(int32_t) * d.E, st)));
  CUtensorMap tu, tc;
  MOE_TRY(make_tmap(&tu, u, false, d.T, d.d, 128));
  MOE_TRY(make_tmap(&tc, cent, false, d.E, d.d, 128));
  const LogitsSplit sp = logits_split(d);
  LogitsArgs a;
  a.T = d.T;
  a.E = d.E;
  a.K = d.d;
  a.kb_per_split = sp.kb_per_split;
  a.z = z;
  a.split_stride = int64_t(d.T) * d.E;
  a.status = status;
  const int64_t grid = cdiv(d.T, 128) * cdiv(d.E, 128) * sp.splits;
  if (grid > INT_MAX) return MOE_ERR_UNSUPPORTED;
  constexpr size_t smem = logits_smem_bytes();
  MOE_TRY(cuda_ok(cudaFuncSetAttribute(logits_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem))));
  logits_gemm_kernel<<<static_cast<unsigned>(grid), 192, smem, st>>>(tu, tc, a);
  MOE_TRY(launched());
  if (rec) MOE_TRY(rec->mark());
  const unsigned blocks = static_cast<unsigned>(cdiv(int64_t(d.T) * 32, 256));
  const int vpl = (d.E + 31) / 32;
#define MOE_TOPK(V)                                                                                              \
  route_topk_kernel<V><<<blocks, 256, 0, st>>>(z, sp.splits, a.split_stride, d.T, d.E, d.k, bias, idx, gate, counts, \
                                               mask, W, d.route_groups > 0 ? d.E / d.route_groups : 0,            \
                                               d.route_group_limit, status)
  if (vpl <= 1) MOE_TOPK(1);
  else if (vpl <= 2) MOE_TOPK(2);
  else if (vpl <= 4) MOE_TOPK(4);
  else if (vpl <= 8) MOE_TOPK(8);
  else if (vpl <= 16) MOE_TOPK(16);
  else MOE_TOPK(32);
#undef MOE_TOPK
  MOE_TRY(launched());
  return rec ? rec->mark() : MOE_OK;
}

// Expert row counts and offsets from the token-expert mask, the GEMM group
// table, and the gather of permuted rows (FP8: quantised on the way).
// Column ranges per token of the gather and the combine: one for large
// batches, more when few tokens would leave most SMs idle (a decode step).
unsigned token_splits(int T, int d) {
  if (T >= 2048) return 1;
  const int chunks = (d / 8 + 127) / 128;  // 128 threads x 16 bytes per range
  return static_cast<unsigned>(chunks < 8 ? (chunks > 0 ? chunks : 1) : 8);
}

moe_status enqueue_dispatch(const moe_dims& d, const int32_t* idx, const uint16_t* u, const uint32_t* mask,
                            int32_t* wprefix, int32_t* cnt, int32_t* offsets, GroupEntry* groups, int32_t* mt_total,
                            int32_t* cgroup, int32_t* perm, int32_t* slot, void* x, float* xs, uint8_t* uq, float* uqs, int* status,
                            cudaStream_t st, Recorder* rec = nullptr, const int32_t* group_weight = nullptr,
                            int n_weights = 0) {
  const int W = (d.T + 31) / 32;
  expert_scan_kernel<<<d.E, 256, 0, st>>>(mask, W, wprefix, cnt);
  MOE_TRY(launched());
  plan_kernel<<<1, 1024, 0, st>>>(cnt, nullptr, d.E, 0, chunk_rows(d), offsets, groups, mt_total, cgroup,
                                  static_cast<int>(cgroup_cap(d)), group_weight, n_weights, status);
  MOE_TRY(launched());
  if (rec) MOE_TRY(rec->mark());
  if (d.T == 0) return rec ? rec->mark() : MOE_OK;  // the offsets (all zero) are the whole result
  const dim3 blocks(static_cast<unsigned>(cdiv(int64_t(d.T) * 32, 256)), token_splits(d.T, d.d));
  const int64_t rows = int64_t(d.T) * d.k;
  const __nv_bfloat16* ub = reinterpret_cast<const __nv_bfloat16*>(u);
  if (is_fp8(d))
    dispatch_kernel<true><<<blocks, 256, 0, st>>>(idx, d.T, d.k, d.E, mask, wprefix, W, offsets, slot, perm, ub, d.d,
                                                  x, xs, rows, uq, uqs, status, d.prec == MOE_FP8_UE8M0);
  else
    dispatch_kernel<false><<<blocks, 256, 0, st>>>(idx, d.T, d.k, d.E, mask, wprefix, W, offsets, slot, perm, ub,
                                                   d.d, x, nullptr, rows, nullptr, nullptr, status, false);
  MOE_TRY(launched());
  return rec ? rec->mark() : MOE_OK;
}

// Streaming multiprocessors of the current device (the persistent grid).
moe_status sm_count(int* n) {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) {
    *n = cache[dev];
    return MOE_OK;
  }
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return MOE_ERR_CUDA;
  if (dev >= 0 && dev < 64) cache[dev] = v;
  *n = v;
  return MOE_OK;
}

template <Epi EPI, bool WIDE>
moe_status launch_xgemm(const CUtensorMap& tw, const CUtensorMap& tx, const XGemmArgs& a, int64_t items_bound,
                        cudaStream_t st) {
  if (items_bound <= 0) return MOE_OK;
  int sms = 0;
  MOE_TRY(sm_count(&sms));
  const int64_t grid = items_bound < sms ? items_bound : sms;
  constexpr size_t smem = xgemm_smem_bytes<WIDE>();
  auto kern = expert_gemm_kernel<EPI, WIDE>;
  MOE_TRY(cuda_ok(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))));
  kern<<<static_cast<unsigned>(grid), kXThreads, smem, st>>>(tw, tx, a);
  return launched();
}

template <Epi EPI, int EW, bool POW2>
moe_status launch_fp8_ew(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, int64_t grid,
                         cudaStream_t st) {
  constexpr size_t smem = fp8_gemm_smem_bytes<EPI, EW>();
  auto kern = fp8_gemm_kernel<EPI, EW, POW2>;
  // The kernel moves registers between its warpgroups (setmaxnreg); its split
  // adds up to exactly LAUNCH_REGS per thread, so a build that launched with
  // fewer would leave the epilogue warps waiting for registers forever.
  cudaFuncAttributes fa;
  MOE_TRY(cuda_ok(cudaFuncGetAttributes(&fa, kern)));
  if (fa.numRegs != F8Shape<EW>::LAUNCH_REGS) return MOE_ERR_CUDA;
  MOE_TRY(cuda_ok(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))));
  kern<<<static_cast<unsigned>(grid), F8Shape<EW>::THREADS, smem, st>>>(ta, tb, a);
  return launched();
}

// few_rows: most 128-row tiles hold few valid rows (fewer than 64 rows per
// group on average), so the work sits on one TMEM lane quarter: 16 epilogue
// warps share it.
template <Epi EPI>
moe_status launch_fp8(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, int64_t items_bound,
                      bool few_rows, bool pow2, cudaStream_t st) {
  if (items_bound <= 0) return MOE_OK;
  int sms = 0;
  MOE_TRY(sm_count(&sms));
  const int64_t grid = items_bound < sms ? items_bound : sms;
  if constexpr (EPI == Epi::SWIGLU) {  // only the SwiGLU epilogue quantises (h), so only it has UE8M0 variants
    if (pow2)
      return few_rows ? launch_fp8_ew<EPI, 16, true>(ta, tb, a, grid, st) : launch_fp8_ew<EPI, 8, true>(ta, tb, a, grid, st);
  }
  return few_rows ? launch_fp8_ew<EPI, 16, false>(ta, tb, a, grid, st) : launch_fp8_ew<EPI, 8, false>(ta, tb, a, grid, st);
}

// Gate/up (+SwiGLU) then down GEMMs over a set of groups.
//   table != nullptr: routed experts, rows from the device table (chunk
//   counts from plan_kernel with chunk_rows(d); upper bound rows_cap rows over
//   n_groups groups).  Otherwise n_groups uniform groups of uni_m rows each;
//   gate/up X rows start at 0 for every group (all shared experts read the
//   same tokens).
struct FfnOperands {
  const void* x;
  const float* xs;
  int64_t x_rows;  // rows allocated in x
  const void* w13;
  const float* w13s;
  const void* w2;
  const float* w2s;
  void* h;
  float* hs;
  uint16_t* y;
  int64_t rows_cap;  // rows allocated in h and y
  const int32_t* group_weight = nullptr;  // table groups -> experts of the weight arrays (nullptr: g -> g)
  int32_t n_weights = 0;                  // experts in the weight arrays when group_weight is given
};

// Experts held in the weight arrays of a launch over n_groups groups.
int64_t weight_experts(const FfnOperands& o, int n_groups) { return o.group_weight ? o.n_weights : n_groups; }

// FP8: tokens on the 128 TMEM lanes (128-row tiles of grouped_gemm_kernel),
// so the promotion scale of a lane is one activation scale per k-block.
moe_status enqueue_ffn_fp8(const moe_dims& d, const FfnOperands& o, int n_groups, const GroupEntry* table,
                           const int32_t* mt_total, const int32_t* cgroup, int uni_m, int* queue, int* status,
                           cudaStream_t st, Recorder* rec) {
  const int I = d.inter, D = d.d;
  CUtensorMap ta1, tb1, ta2, tb2;
  MOE_TRY(make_tmap(&ta1, o.x, true, o.x_rows, D, 128));
  MOE_TRY(make_tmap(&tb1, o.w13, true, weight_experts(o, n_groups) * 2 * I, D, 256));
  MOE_TRY(make_tmap(&ta2, o.h, true, o.rows_cap, I, 128));
  MOE_TRY(make_tmap(&tb2, o.w2, true, weight_experts(o, n_groups) * D, I, 256));
  const int64_t mt = table ? cdiv(o.rows_cap + 127 * int64_t(n_groups), 128) : int64_t(n_groups) * cdiv(uni_m, 128);

  GemmArgs a = base_args(status);
  a.queue = queue;
  a.groups = table;
  a.mt_total = mt_total;
  a.chunk_group = cgroup;
  a.n_groups = n_groups;
  a.uni_m = uni_m;
  a.uni_a_step = 0;
  a.uni_out_step = uni_m;
  a.N = 2 * I;
  a.K = D;
  a.b_rows_per_group = 2 * I;
  a.a_rows_cap = static_cast<int32_t>(o.x_rows);
  a.out = o.h;
  a.out_ld = I;
  a.a_scale = o.xs;
  a.a_scale_ld = o.x_rows;
  a.b_scale = o.w13s;
  a.out_scale = o.hs;
  a.out_scale_ld = o.rows_cap;
#ifdef MOE_CHECK
  a.b_rows = weight_experts(o, n_groups) * 2 * I;
  a.out_rows = static_cast<int32_t>(o.rows_cap);
#endif
  const bool few_rows = (table ? o.rows_cap : int64_t(uni_m) * n_groups) < 64 * int64_t(n_groups);
  MOE_TRY((launch_fp8<Epi::SWIGLU>(ta1, tb1, a, mt * (2 * I / 256), few_rows, d.prec == MOE_FP8_UE8M0, st)));
  if (rec) MOE_TRY(rec->mark());

  GemmArgs b = a;
  b.queue = queue + 1;
  b.uni_a_step = uni_m;
  b.N = D;
  b.K = I;
  b.b_rows_per_group = D;
  b.a_rows_cap = static_cast<int32_t>(o.rows_cap);
  b.out = o.y;
  b.out_ld = D;
  b.a_scale = o.hs;
  b.a_scale_ld = o.rows_cap;
  b.b_scale = o.w2s;
  b.out_scale = nullptr;
#ifdef MOE_CHECK
  b.b_rows = weight_experts(o, n_groups) * D;
#endif
  MOE_TRY((launch_fp8<Epi::BF16>(ta2, tb2, b, mt * cdiv(D, 256), few_rows, false, st)));
  return rec ? rec->mark() : MOE_OK;
}

// bf16: weights on the TMEM lanes, tokens on the columns (expert_gemm_kernel).
// queue: two zeroed item counters (gate/up launch, down launch).
moe_status enqueue_ffn(const moe_dims& d, const FfnOperands& o, int n_groups, const GroupEntry* table,
                       const int32_t* ch_total, const int32_t* cgroup, int uni_m, int* queue, int* status,
                       cudaStream_t st, Recorder* rec = nullptr) {
  if (is_fp8(d))
    return enqueue_ffn_fp8(d, o, n_groups, table, ch_total, cgroup, uni_m, queue, status, st, rec);
  const int I = d.inter, D = d.d;
  // Kernel shapes (XShape), measured: both GEMMs of the shared experts (every
  // token: many chunks per weight block) run wide; the routed gate/up GEMM runs
  // narrow; the routed down GEMM runs wide when the launch has many wide items
  // per SM (V3: ~70, 3-8% faster), else narrow (mid and a 32-expert slice,
  // under 10 per SM: the longer wide items leave a longer tail, 8-13% slower).
  int sms = 0;
  MOE_TRY(sm_count(&sms));
  constexpr int CH_N = XShape<false>::CH, CH_W = XShape<true>::CH;
  const bool up_wide = table == nullptr;
  const bool down_wide = table == nullptr || (o.rows_cap / CH_W + n_groups / 2) * cdiv(D, 256) >= int64_t(24) * sms;
  CUtensorMap tx1, tw1, tx2, tw2;
  MOE_TRY(make_tmap(&tx1, o.x, false, o.x_rows, D, up_wide ? CH_W : CH_N));
  MOE_TRY(make_tmap(&tw1, o.w13, false, weight_experts(o, n_groups) * 2 * I, D, 256));
  MOE_TRY(make_tmap(&tx2, o.h, false, o.rows_cap, I, down_wide ? CH_W : CH_N));
  MOE_TRY(make_tmap(&tw2, o.w2, false, weight_experts(o, n_groups) * D, I, 256));
  // upper bound of the items per weight block: a table's 128-row chunks (every
  // group adds at most one partial chunk; the wide kernel walks the same
  // table), or the uniform groups' items of the launch's shape
  const int64_t table_chunks = cdiv(o.rows_cap + int64_t(kChunkBf16 - 1) * n_groups, kChunkBf16);
  const int64_t items_up = table ? table_chunks : int64_t(n_groups) * cdiv(uni_m, up_wide ? CH_W : CH_N);
  const int64_t items_down = table ? table_chunks : int64_t(n_groups) * cdiv(uni_m, down_wide ? CH_W : CH_N);

  XGemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.status = status;
  a.queue = queue;
  a.groups = table;
  a.ch_total = ch_total;
  a.chunk_group = cgroup;
  a.n_groups = n_groups;
  a.uni_m = uni_m;
  a.uni_a_step = 0;
  a.uni_out_step = uni_m;
  a.Nw = 2 * I;
  a.K = D;
  a.x_rows = static_cast<int32_t>(o.x_rows);
  a.out = o.h;
  a.out_ld = I;
#ifdef MOE_CHECK
  a.w_rows = weight_experts(o, n_groups) * 2 * I;
  a.out_rows = static_cast<int32_t>(o.rows_cap);
#endif
  if (up_wide) MOE_TRY((launch_xgemm<Epi::SWIGLU, true>(tw1, tx1, a, items_up * cdiv(2 * I, 256), st)));
  else MOE_TRY((launch_xgemm<Epi::SWIGLU, false>(tw1, tx1, a, items_up * cdiv(2 * I, 256), st)));
  if (rec) MOE_TRY(rec->mark());

  XGemmArgs b = a;
  b.queue = queue + 1;
  b.uni_a_step = uni_m;
  b.Nw = D;
  b.K = I;
  b.x_rows = static_cast<int32_t>(o.rows_cap);
  b.out = o.y;
  b.out_ld = D;
#ifdef MOE_CHECK
  b.w_rows = weight_experts(o, n_groups) * D;
#endif
  if (down_wide) MOE_TRY((launch_xgemm<Epi::BF16, true>(tw2, tx2, b, items_down * cdiv(D, 256), st)));
  else MOE_TRY((launch_xgemm<Epi::BF16, false>(tw2, tx2, b, items_down * cdiv(D, 256), st)));
  return rec ? rec->mark() : MOE_OK;
}

moe_status check_weights(const moe_dims& d, const moe_weights* w) {
  if (!w || !w->w13 || !w->w2 || !w->centroids) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w->w13) || !aligned16(w->w2) || !aligned16(w->centroids)) return MOE_ERR_INVALID_ARG;
  if (d.n_shared > 0 && (!w->ws13 || !w->ws2 || !aligned16(w->ws13) || !aligned16(w->ws2))) return MOE_ERR_INVALID_ARG;
  if (is_fp8(d)) {
    if (!w->w13_scale || !w->w2_scale) return MOE_ERR_INVALID_ARG;
    if (d.n_shared > 0 && (!w->ws13_scale || !w->ws2_scale)) return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

}  // namespace

// =================================================================== C ABI
extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_BAD_INDEX: return "expert index or offset out of range";
    case MOE_ERR_OUT_OF_RANGE: return "index outside its buffer (range-checked build)";
  }
  return "unknown status";
}

moe_status moe_workspace_size(const moe_dims* dims, size_t* bytes) {
  MOE_TRY(check_dims(dims));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_layout(*dims).total;
  return MOE_OK;
}

moe_status moe_route(const moe_dims* dims, const uint16_t* u, const uint16_t* centroids, const float* bias,
                     int32_t* topk_idx, float* topk_gate, int32_t* counts, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_dims(dims));
  MOE_TRY(check_ws(dims, ws, ws_bytes));
  // token-sized buffers may be empty (null) when T == 0
  const bool empty = dims->T == 0;
  if (!centroids || !bias || !counts || (!empty && (!u || !topk_idx || !topk_gate))) return MOE_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(centroids)) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*dims);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_TRY(cuda_ok(cudaMemsetAsync(at<int>(ws, L.status), 0, sizeof(int), st)));
  if (dims->T == 0) return cuda_ok(cudaMemsetAsync(counts, 0, sizeof(int32_t) * dims->E, st));
  return enqueue_route(*dims, u, centroids, bias, topk_idx, topk_gate, counts, nullptr, at<float>(ws, L.z),
                       at<int>(ws, L.status), st);
}

moe_status moe_permute(const moe_dims* dims, const int32_t* topk_idx, const uint16_t* u, int32_t* offsets,
                       int32_t* perm, int32_t* slot, void* x_perm, float* x_scale, void* ws, size_t ws_bytes,
                       void* stream) {
  MOE_TRY(check_dims(dims));
  MOE_TRY(check_ws(dims, ws, ws_bytes));
  // token-sized buffers may be empty (null) when T == 0
  const bool empty = dims->T == 0;
  if (!offsets || (!empty && (!topk_idx || !u || !perm || !slot || !x_perm))) return MOE_ERR_INVALID_ARG;
  if (is_fp8(*dims) && !empty && !x_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*dims);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = at<int>(ws, L.status);
  MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, sizeof(int), st)));
  const int W = (dims->T + 31) / 32;
  uint32_t* mask = at<uint32_t>(ws, L.mask);
  MOE_TRY(cuda_ok(cudaMemsetAsync(mask, 0, sizeof(uint32_t) * size_t(dims->E) * W, st)));
  const int64_t n = int64_t(dims->T) * dims->k;
  if (n > 0) {
    build_mask_kernel<<<static_cast<unsigned>(cdiv(n, 256)), 256, 0, st>>>(topk_idx, n, dims->k, dims->E, mask, W,
                                                                           status);
    MOE_TRY(launched());
  }
  return enqueue_dispatch(*dims, topk_idx, u, mask, at<int32_t>(ws, L.wprefix), at<int32_t>(ws, L.cnt), offsets,
                          at<GroupEntry>(ws, L.groups), at<int32_t>(ws, L.mt_total), at<int32_t>(ws, L.cgroup), perm,
                          slot, x_perm, x_scale, nullptr, nullptr, status, st);
}

moe_status moe_grouped_ffn(const moe_dims* dims, int32_t n_groups, int32_t rows, const int32_t* offsets,
                           const int32_t* group_expert, int32_t n_weight_experts, const void* x,
                           const float* x_scale, const void* w13, const float* w13_scale, const void* w2,
                           const float* w2_scale, uint16_t* y, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_dims(dims));
  MOE_TRY(check_ws(dims, ws, ws_bytes));
  const bool fp8 = is_fp8(*dims);
  if (n_groups <= 0 || n_groups > dims->E + dims->n_shared || rows < 0) return MOE_ERR_INVALID_ARG;
  if (group_expert && n_weight_experts <= 0) return MOE_ERR_INVALID_ARG;
  if (int64_t(rows) > int64_t(dims->T) * dims->k) return MOE_ERR_WORKSPACE;
  if (!offsets || !x || !w13 || !w2 || !y) return MOE_ERR_INVALID_ARG;
  if (fp8 && (!x_scale || !w13_scale || !w2_scale)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13) || !aligned16(w2) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*dims);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = at<int>(ws, L.status);
  MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, sizeof(int), st)));
  if (rows == 0) return MOE_OK;
  GroupEntry* groups = at<GroupEntry>(ws, L.groups);
  int32_t* mt_total = at<int32_t>(ws, L.mt_total);
  int32_t* cgroup = at<int32_t>(ws, L.cgroup);
  int* queue = at<int>(ws, L.queue);
  MOE_TRY(cuda_ok(cudaMemsetAsync(queue, 0, 2 * sizeof(int), st)));
  plan_kernel<<<1, 1024, 0, st>>>(nullptr, offsets, n_groups, rows, chunk_rows(*dims), nullptr, groups, mt_total,
                                  cgroup, static_cast<int>(cgroup_cap(*dims)), group_expert, n_weight_experts, status);
  MOE_TRY(launched());
  FfnOperands o{x, x_scale, rows, w13, w13_scale, w2, w2_scale, at<void>(ws, L.h),
                fp8 ? at<float>(ws, L.hs) : nullptr, y, rows, group_expert, n_weight_experts};
  return enqueue_ffn(*dims, o, n_groups, groups, mt_total, cgroup, 0, queue, status, st);
}

moe_status moe_combine(const moe_dims* dims, const uint16_t* u, const uint16_t* shared_y, const uint16_t* y_perm,
                       const int32_t* slot, const float* topk_gate, uint16_t* out, void* stream) {
  MOE_TRY(check_dims(dims));
  if (dims->T == 0) return MOE_OK;  // nothing to combine; the buffers may be empty (null)
  if (!u || !y_perm || !slot || !topk_gate || !out || (dims->n_shared > 0 && !shared_y)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(y_perm) || !aligned16(out) || (shared_y && !aligned16(shared_y)))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  combine_kernel<<<dim3(static_cast<unsigned>(dims->T), token_splits(dims->T, dims->d)), 128, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(u), reinterpret_cast<const __nv_bfloat16*>(shared_y), dims->n_shared,
      reinterpret_cast<const __nv_bfloat16*>(y_perm), slot, topk_gate, dims->T, dims->d, dims->k,
      int64_t(dims->T) * dims->k, reinterpret_cast<__nv_bfloat16*>(out), nullptr);
  return launched();
}

moe_status moe_bias_update(int32_t E, int32_t T, int32_t k, const int32_t* counts, float gamma, float* bias,
                           void* stream) {
  if (E <= 0 || E > 1024 || T < 0 || k <= 0 || k > E || !counts || !bias) return MOE_ERR_INVALID_ARG;
  bias_update_kernel<<<static_cast<unsigned>(cdiv(E, 256)), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      E, T, k, counts, gamma, bias);
  return launched();
}

moe_status moe_forward(const moe_dims* dims, const moe_weights* w, const uint16_t* u, const float* bias,
                       uint16_t* out, int32_t* counts_out, void* ws, size_t ws_bytes, void* stream) {
  return moe_forward_profiled(dims, w, u, bias, out, counts_out, ws, ws_bytes, stream, nullptr, 0);
}

}  // extern "C"

namespace {

// Copies of hot experts (moe_forward_replicated): device tables of the plan.
struct ReplicaPlan {
  const int32_t* first;        // [E]
  const int32_t* count;        // [E]
  const int32_t* slot_expert;  // [P]
  int32_t P;                   // physical slots
};

// The dims the workspace of a forward is laid out for: with a replica plan
// the per-expert tables hold the P physical slots.
moe_dims ws_dims(const moe_dims& d, const ReplicaPlan* rp) {
  moe_dims w = d;
  if (rp && rp->P > w.E) w.E = rp->P;
  return w;
}

moe_status forward_impl(const moe_dims* dims, const moe_weights* w, const uint16_t* u, const float* bias,
                        uint16_t* out, int32_t* counts_out, void* ws, size_t ws_bytes, void* stream,
                        void* const* events, int32_t n_events, const ReplicaPlan* rp) {
  MOE_TRY(check_dims(dims));
  const moe_dims wd = ws_dims(*dims, rp);
  MOE_TRY(check_ws(&wd, ws, ws_bytes));
  MOE_TRY(check_weights(*dims, w));
  // u and out may be empty (null) when T == 0
  if (!bias || (d_T_nonzero(dims) && (!u || !out)) || !aligned16(u) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (events && n_events < MOE_PROFILE_EVENTS) return MOE_ERR_INVALID_ARG;
  const moe_dims& d = *dims;
  const bool fp8 = is_fp8(d);
  const Layout L = make_layout(wd);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Recorder recorder;
  recorder.ev = events;
  recorder.n = n_events;
  recorder.st = st;
  Recorder* rec = events ? &recorder : nullptr;
  if (rec) MOE_TRY(rec->mark());
  int* status = at<int>(ws, L.status);
  int* queue = at<int>(ws, L.queue);
  MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, L.queue + 4 * sizeof(int), st)));  // status word and item counters
  int32_t* counts = counts_out ? counts_out : at<int32_t>(ws, L.counts);
  if (d.T == 0) return cuda_ok(cudaMemsetAsync(counts, 0, sizeof(int32_t) * d.E, st));
  const int W = (d.T + 31) / 32;
  uint32_t* mask = at<uint32_t>(ws, L.mask);
  MOE_TRY(cuda_ok(cudaMemsetAsync(mask, 0, sizeof(uint32_t) * size_t(wd.E) * W, st)));

  int32_t* idx = at<int32_t>(ws, L.idx);
  float* gate = at<float>(ws, L.gate);
  // with copies of hot experts the dispatch mask is over physical slots, set
  // by the replica assignment instead of the router
  MOE_TRY(enqueue_route(d, u, w->centroids, bias, idx, gate, counts, rp ? nullptr : mask, at<float>(ws, L.z), status,
                        st, rec));
  const int64_t R = int64_t(d.T) * d.k;
  moe_dims dd = d;  // the dispatch's view: one group per physical slot
  if (rp) {
    assign_replicas_kernel<<<static_cast<unsigned>(cdiv(R, 256)), 256, 0, st>>>(idx, R, d.k, d.E, rp->first, rp->count,
                                                                                rp->P, mask, W, status);
    MOE_TRY(launched());
    dd.E = rp->P;
  }

  GroupEntry* groups = at<GroupEntry>(ws, L.groups);
  int32_t* mt_total = at<int32_t>(ws, L.mt_total);
  int32_t* slot = at<int32_t>(ws, L.slot);
  MOE_TRY(enqueue_dispatch(dd, idx, u, mask, at<int32_t>(ws, L.wprefix), at<int32_t>(ws, L.cnt),
                           at<int32_t>(ws, L.offsets), groups, mt_total, at<int32_t>(ws, L.cgroup),
                           at<int32_t>(ws, L.perm), slot,
                           at<void>(ws, L.x), fp8 ? at<float>(ws, L.xs) : nullptr,
                           fp8 ? at<uint8_t>(ws, L.uq) : nullptr, fp8 ? at<float>(ws, L.uqs) : nullptr, status, st,
                           rec, rp ? rp->slot_expert : nullptr, d.E));

  // routed experts: groups from the device table
  FfnOperands ro{at<void>(ws, L.x), fp8 ? at<float>(ws, L.xs) : nullptr, R, w->w13, w->w13_scale, w->w2,
                 w->w2_scale, at<void>(ws, L.h), fp8 ? at<float>(ws, L.hs) : nullptr, at<uint16_t>(ws, L.y), R,
                 rp ? rp->slot_expert : nullptr, d.E};
  MOE_TRY(enqueue_ffn(d, ro, dd.E, groups, mt_total, at<int32_t>(ws, L.cgroup), 0, queue, status, st, rec));

  // shared experts: every token, n_shared uniform groups
  uint16_t* ysh = at<uint16_t>(ws, L.ysh);
  if (d.n_shared > 0) {
    const void* xa = fp8 ? static_cast<const void*>(at<uint8_t>(ws, L.uq)) : static_cast<const void*>(u);
    FfnOperands so{xa, fp8 ? at<float>(ws, L.uqs) : nullptr, d.T, w->ws13, w->ws13_scale, w->ws2, w->ws2_scale,
                   at<void>(ws, L.hsh), fp8 ? at<float>(ws, L.hshs) : nullptr, ysh, int64_t(d.n_shared) * d.T};
    MOE_TRY(enqueue_ffn(d, so, d.n_shared, nullptr, nullptr, nullptr, d.T, queue + 2, status, st, rec));
  } else if (rec) {
    MOE_TRY(rec->mark());
    MOE_TRY(rec->mark());
  }

  combine_kernel<<<dim3(static_cast<unsigned>(d.T), token_splits(d.T, d.d)), 128, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(u), reinterpret_cast<const __nv_bfloat16*>(ysh), d.n_shared,
      at<const __nv_bfloat16>(ws, L.y), slot, gate, d.T, d.d, d.k, R, reinterpret_cast<__nv_bfloat16*>(out), status);
  MOE_TRY(launched());
  return rec ? rec->mark() : MOE_OK;
}

}  // namespace

// =================================================================== backward (bf16)
namespace {

// Backward workspace: the forward's layout (routing, dispatch, x_perm, h, y)
// followed by the backward's own buffers.
struct BwdLayout {
  Layout f;
  size_t queue, ab, dy, dh, dab, dx, dz_row, ab_s, dh_s, dab_s, dx_s, pad_off, row_of_col, wg_r, wg_s2, wg_s13;
  size_t xT, dyT, hT, dabT, uT, GT, hsT, dabsT;
  // FP8 only: bf16 h (routed, shared) and the E4M3 codes + 1 x 128 scales of
  // the data-gradient GEMMs' activation operands
  size_t hb, hsb, dyq, dys, dabq, dabs, Gq, Gs, dabsq, dabss, total;
  int64_t Rp, Tp;
};

BwdLayout make_bwd_layout(const moe_dims& d) {
  BwdLayout B{};
  B.f = make_layout(d);
  size_t off = B.f.total;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes > 0 ? bytes : 1);
    return o;
  };
  const int64_t T = d.T, R = T * d.k, E = d.E, I = d.inter, D = d.d, Ns = d.n_shared;
  // every expert's rows padded to a multiple of 64 columns (FP8: 128, the
  // token blocks of the weight-gradient operands' quantisation)
  const int64_t gran = is_fp8(d) ? 128 : 64;
  B.Rp = (R + gran * E + gran - 1) / gran * gran;
  B.Tp = (T + gran - 1) / gran * gran;
  B.queue = take(16 * sizeof(int));
  B.ab = take(R * 2 * I * 2);
  B.dy = take(R * D * 2);
  B.dh = take(R * I * 2);
  B.dab = take(R * 2 * I * 2);
  B.dx = take(R * D * 2);
  B.dz_row = take(R * 4);
  B.ab_s = take(Ns * T * 2 * I * 2);
  B.dh_s = take(Ns * T * I * 2);
  B.dab_s = take(Ns * T * 2 * I * 2);
  B.dx_s = take(Ns * T * D * 2);
  B.pad_off = take((E + 2) * 4);
  B.row_of_col = take(B.Rp * 4);
  B.wg_r = take(E * sizeof(WgradGroup));
  B.wg_s2 = take((Ns + 1) * sizeof(WgradGroup));
  B.wg_s13 = take((Ns + 1) * sizeof(WgradGroup));
  B.xT = take(D * B.Rp * 2);
  B.dyT = take(D * B.Rp * 2);
  B.hT = take(I * B.Rp * 2);
  B.dabT = take(2 * I * B.Rp * 2);
  B.uT = take(D * B.Tp * 2);
  B.GT = take(D * B.Tp * 2);
  B.hsT = take(I * Ns * B.Tp * 2);
  B.dabsT = take(2 * I * Ns * B.Tp * 2);
  if (is_fp8(d)) {
    B.hb = take(R * I * 2);
    B.hsb = take(Ns * T * I * 2);
    B.dyq = take(R * D);
    B.dys = take(D / 128 * R * 4);
    B.dabq = take(R * 2 * I);
    B.dabs = take(2 * I / 128 * R * 4);
    B.Gq = take(T * D);
    B.Gs = take(D / 128 * T * 4);
    B.dabsq = take(Ns * T * 2 * I);
    B.dabss = take(2 * I / 128 * Ns * T * 4);
  }
  B.total = off;
  return B;
}

// WgradGroup table of the routed experts from the padded offsets: the same
// K range in A and B.
__global__ void wgrad_table_kernel(const int32_t* __restrict__ pad_off, int G, WgradGroup* __restrict__ out) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g < G) out[g] = WgradGroup{pad_off[g], pad_off[g], pad_off[g + 1] - pad_off[g], 0};
}

// WgradGroup table of the shared experts: group s reads K columns
// [s * a_step, + len) of A and [s * b_step, + len) of B.
__global__ void wgrad_strided_table_kernel(int G, int a_step, int b_step, int len, WgradGroup* __restrict__ out) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g < G) out[g] = WgradGroup{g * a_step, g * b_step, len, 0};
}

// One bf16 expert-GEMM launch (BF16 epilogue): out[rows of group g] = X[rows] . W_g^T,
// on the narrow or the wide kernel shape (XShape).
//   table != nullptr: groups from the device table (chunk totals in mt_total,
//   chunk -> group in cgroup); else n_groups uniform groups of uni_m rows,
//   X rows of group g starting at g * uni_a_step, output rows at g * uni_m.
moe_status xgemm_bf16(const void* w, int64_t w_rows, int Nw, int K, const void* x, int64_t x_rows, void* out,
                      int64_t out_ld, int n_groups, const GroupEntry* table, const int32_t* mt_total,
                      const int32_t* cgroup, int64_t chunks_bound, int uni_m, int uni_a_step, int* queue, int* status,
                      bool wide, cudaStream_t st) {
  CUtensorMap tw, tx;
  MOE_TRY(make_tmap(&tw, w, false, w_rows, K, 256));
  MOE_TRY(make_tmap(&tx, x, false, x_rows, K, wide ? XShape<true>::CH : XShape<false>::CH));
  XGemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.status = status;
  a.queue = queue;
  a.groups = table;
  a.ch_total = mt_total;
  a.chunk_group = cgroup;
  a.n_groups = n_groups;
  a.uni_m = uni_m;
  a.uni_a_step = uni_a_step;
  a.uni_out_step = uni_m;
  a.Nw = Nw;
  a.K = K;
  a.x_rows = static_cast<int32_t>(x_rows);
  a.out = out;
  a.out_ld = out_ld;
#ifdef MOE_CHECK
  a.w_rows = w_rows;
  a.out_rows = static_cast<int32_t>(table ? x_rows : int64_t(uni_m) * n_groups);
#endif
  const int64_t chunks =
      table ? chunks_bound : int64_t(n_groups) * cdiv(uni_m, wide ? XShape<true>::CH : XShape<false>::CH);
  if (wide) return launch_xgemm<Epi::BF16, true>(tw, tx, a, chunks * cdiv(Nw, 256), st);
  return launch_xgemm<Epi::BF16, false>(tw, tx, a, chunks * cdiv(Nw, 256), st);
}

// Transposed gather src [batch][rows][C] -> dst [batch][C][n_cols] (row ldd)
// of transpose_cols_kernel: dst column col holds src row row_of_col[col]
// (through perm when given; -1: zeros), or row col while col < rows when
// row_of_col is null; with n_live (a device count) only the columns below it.
// FQ: the FP8 weight-gradient operands, quantised 1 x 128 along the columns
// and dequantised to bf16.
template <bool FQ>
moe_status transpose_cols(const void* src, int rows, int C, int64_t src_batch, const int32_t* row_of_col,
                          const int32_t* perm, const int32_t* n_live, int64_t n_cols, void* dst, int64_t ldd,
                          int64_t dst_batch, int batch, bool pow2, cudaStream_t st) {
  if (n_cols <= 0 || C <= 0 || batch <= 0) return MOE_OK;
  if (C % 8 || ldd % (FQ ? 8 : 2) || n_cols > INT_MAX || (reinterpret_cast<uintptr_t>(dst) & (FQ ? 15 : 3)))
    return MOE_ERR_UNSUPPORTED;
  // enough blocks for ~16 per SM; each walks n_slab / split slabs of 64 c
  const int64_t col_tiles = cdiv(n_cols, 128) * batch, n_slab = cdiv(C, 64);
  const int64_t split = std::min<int64_t>(n_slab, std::max<int64_t>(1, cdiv(int64_t(148) * 16, col_tiles)));
  dim3 grid(static_cast<unsigned>(split), static_cast<unsigned>(cdiv(n_cols, 128)), static_cast<unsigned>(batch));
  transpose_cols_kernel<FQ><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), rows, C, src_batch,
                                                  row_of_col, perm, static_cast<int>(n_cols), n_live,
                                                  static_cast<__nv_bfloat16*>(dst), ldd, dst_batch, pow2);
  return launched();
}

moe_status transpose_bf16(const void* src, int rows, int C, int64_t src_batch, const int32_t* row_of_col,
                          const int32_t* n_live, int64_t n_cols, void* dst, int64_t ldd, int64_t dst_batch, int batch,
                          cudaStream_t st) {
  return transpose_cols<false>(src, rows, C, src_batch, row_of_col, nullptr, n_live, n_cols, dst, ldd, dst_batch,
                               batch, false, st);
}

moe_status transpose_fq(const void* src, int rows, int C, int64_t src_batch, const int32_t* row_of_col,
                        const int32_t* perm, const int32_t* n_live, int64_t n_cols, void* dst, int64_t ldd,
                        int64_t dst_batch, int batch, bool pow2, cudaStream_t st) {
  return transpose_cols<true>(src, rows, C, src_batch, row_of_col, perm, n_live, n_cols, dst, ldd, dst_batch, batch,
                              pow2, st);
}

// 1 x 128 quantisation of bf16 rows [rows, C] -> codes + scales [C/128][scale_ld].
moe_status quant_rows(const void* src, int64_t rows, int C, void* codes, void* scales, int64_t scale_ld, bool pow2,
                      cudaStream_t st) {
  if (rows <= 0) return MOE_OK;
  quant_rows_kernel<<<static_cast<unsigned>(cdiv(rows * 32, 256)), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(src), rows, C, static_cast<uint8_t*>(codes), static_cast<float*>(scales),
      scale_ld, pow2);
  return launched();
}

// One FP8 expert-GEMM launch with the bf16 epilogue: out[rows of group g] =
// dequant(A rows) . dequant(W_g)^T, A codes [a_rows, K] with 1 x 128 scales
// [K/128][a_scale_ld], W codes [.. , K] with N rows per group and 128 x 128
// block scales.  table != nullptr: groups from the device tables (rows_cap
// rows at most); else n_groups uniform groups of uni_m rows, A rows of group
// g from g * uni_a_step, output rows from g * uni_m.
moe_status fp8gemm_bf16(const void* w, const float* wsc, int64_t w_rows, int N, int K, const void* a,
                        const float* asc, int64_t a_scale_ld, int64_t a_rows, void* out, int64_t out_ld, int n_groups,
                        const GroupEntry* table, const int32_t* mt_total, const int32_t* cgroup, int64_t rows_cap,
                        int uni_m, int uni_a_step, int* queue, int* status, cudaStream_t st) {
  CUtensorMap ta, tb;
  MOE_TRY(make_tmap(&ta, a, true, a_rows, K, 128));
  MOE_TRY(make_tmap(&tb, w, true, w_rows, K, 256));
  GemmArgs g = base_args(status);
  g.queue = queue;
  g.groups = table;
  g.mt_total = mt_total;
  g.chunk_group = cgroup;
  g.n_groups = n_groups;
  g.uni_m = uni_m;
  g.uni_a_step = uni_a_step;
  g.uni_out_step = uni_m;
  g.N = N;
  g.K = K;
  g.b_rows_per_group = N;
  g.a_rows_cap = static_cast<int32_t>(a_rows);
  g.out = out;
  g.out_ld = out_ld;
  g.a_scale = asc;
  g.a_scale_ld = a_scale_ld;
  g.b_scale = wsc;
  const int64_t rows = table ? rows_cap : int64_t(uni_m) * n_groups;
#ifdef MOE_CHECK
  g.b_rows = w_rows;
  g.out_rows = static_cast<int32_t>(rows);
#endif
  const int64_t mt = table ? cdiv(rows_cap + 127 * int64_t(n_groups), 128) : int64_t(n_groups) * cdiv(uni_m, 128);
  return launch_fp8<Epi::BF16>(ta, tb, g, mt * cdiv(N, 256), rows < 64 * int64_t(n_groups), false, st);
}

// Weight gradients of n_groups groups: out[g] [M, N] fp32 = A[:, ka..] . B[:, kb..]^T.
// fp32 output [G][M][N] for TMA stores: boxes of 32 x 32 elements, 128-byte
// swizzle (the layout the wgrad epilogue writes its staging boxes in).
moe_status make_tmap_out3d(CUtensorMap* map, float* base, int64_t G, int64_t M, int64_t N) {
  auto fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(G)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(N * 4), static_cast<cuuint64_t>(M * N * 4)};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// Weight gradients out[g] = A[:, ka_g ..] . B[:, kb_g ..]^T for n_groups groups
// (persistent wgrad_gemm_kernel; queue: one zeroed item counter).
moe_status wgrad(const void* A, int64_t a_cols, int M, const void* Bm, int64_t b_cols, int N,
                 const WgradGroup* table, int n_groups, float* out, int* queue, int* status, cudaStream_t st) {
  if (n_groups <= 0) return MOE_OK;
  if (N % 4) return MOE_ERR_UNSUPPORTED;  // fp32 rows of the output map: 16-byte multiples
  CUtensorMap ta, tb, to;
  MOE_TRY(make_tmap(&ta, A, false, M, a_cols, 128));
  MOE_TRY(make_tmap(&tb, Bm, false, N, b_cols, 256));
  MOE_TRY(make_tmap_out3d(&to, out, n_groups, M, N));
  WgradArgs a{table, n_groups, M, N, static_cast<int32_t>(cdiv(M, 128)), static_cast<int32_t>(cdiv(N, 256)), queue,
              status};
  const int64_t items = int64_t(n_groups) * a.m_tiles * a.n_tiles;
  if (items > INT_MAX) return MOE_ERR_UNSUPPORTED;
  int sms = 0;
  MOE_TRY(sm_count(&sms));
  const int64_t grid = items < sms ? items : sms;
  constexpr size_t smem = wgrad_smem_bytes();
  MOE_TRY(cuda_ok(cudaFuncSetAttribute(wgrad_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem))));
  wgrad_gemm_kernel<<<static_cast<unsigned>(grid), kWgThreads, smem, st>>>(ta, tb, to, a);
  return launched();
}

unsigned ew_blocks(int64_t n) {  // grid of the elementwise kernels (grid-strided)
  const int64_t b = cdiv(n, 256);
  return static_cast<unsigned>(b < 148 * 16 ? (b > 0 ? b : 1) : 148 * 16);
}

// The backward pass in the FP8 scheme after the routing (idx, gate, z, the
// token x expert mask are in the workspace): see moe_backward in moe.h.
moe_status backward_fp8(const moe_dims& d, const BwdLayout& B, const moe_weights* w, const moe_weights_t* wt,
                        const uint16_t* u, const uint16_t* dout, const moe_grads* gr, void* ws, cudaStream_t st) {
  const Layout& L = B.f;
  const int64_t T = d.T, R = T * d.k, E = d.E, I = d.inter, D = d.d, Ns = d.n_shared, I2 = 2 * I;
  const bool pow2 = d.prec == MOE_FP8_UE8M0;
  int* status = at<int>(ws, L.status);
  int* queue = at<int>(ws, B.queue);
  int32_t* idx = at<int32_t>(ws, L.idx);
  float* gate = at<float>(ws, L.gate);
  float* z = at<float>(ws, L.z);
  GroupEntry* groups = at<GroupEntry>(ws, L.groups);
  int32_t* mt_total = at<int32_t>(ws, L.mt_total);
  int32_t* cgroup = at<int32_t>(ws, L.cgroup);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* perm = at<int32_t>(ws, L.perm);
  int32_t* slot = at<int32_t>(ws, L.slot);
  void* x = at<void>(ws, L.x);       // E4M3 codes of the routed rows, scales xs [d/128][R]
  float* xs = at<float>(ws, L.xs);
  uint8_t* uq = Ns > 0 ? at<uint8_t>(ws, L.uq) : nullptr;  // codes of u for the shared experts, uqs [d/128][T]
  float* uqs = Ns > 0 ? at<float>(ws, L.uqs) : nullptr;
  MOE_TRY(enqueue_dispatch(d, idx, u, at<uint32_t>(ws, L.mask), at<int32_t>(ws, L.wprefix), at<int32_t>(ws, L.cnt),
                           offsets, groups, mt_total, cgroup, perm, slot, x, xs, uq, uqs, status, st));
  const int Ei = static_cast<int>(E), Nsi = static_cast<int>(Ns), Ti = static_cast<int>(T);
  void* ab = at<void>(ws, B.ab);
  void* hb = at<void>(ws, B.hb);
  void* hq = at<void>(ws, L.h);
  float* hs = at<float>(ws, L.hs);
  void* y = at<void>(ws, L.y);
  // --- routed experts, forward: a|b (bf16), h (bf16, then E4M3 along I), y
  MOE_TRY(fp8gemm_bf16(w->w13, w->w13_scale, E * I2, static_cast<int>(I2), static_cast<int>(D), x, xs, R, R, ab, I2,
                       Ei, groups, mt_total, cgroup, R, 0, 0, queue + 0, status, st));
  swiglu_fwd_kernel<<<ew_blocks(R * I / 8), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(ab), R,
                                                           static_cast<int>(I), static_cast<__nv_bfloat16*>(hb));
  MOE_TRY(launched());
  MOE_TRY(quant_rows(hb, R, static_cast<int>(I), hq, hs, R, pow2, st));
  MOE_TRY(fp8gemm_bf16(w->w2, w->w2_scale, E * D, static_cast<int>(D), static_cast<int>(I), hq, hs, R, R, y, D, Ei,
                       groups, mt_total, cgroup, R, 0, 0, queue + 1, status, st));
  // --- combine and gates backward (fp32): dy, dz, du = G + router share
  void* dy = at<void>(ws, B.dy);
  float* dz_row = at<float>(ws, B.dz_row);
  const LogitsSplit sp = logits_split(d);
  combine_bwd_kernel<<<static_cast<unsigned>(T), 128, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(dout), static_cast<const __nv_bfloat16*>(y), slot, idx, gate, z,
      sp.splits, T * E, reinterpret_cast<const __nv_bfloat16*>(w->centroids), Ti, static_cast<int>(D), d.k, Ei, R,
      static_cast<__nv_bfloat16*>(dy), dz_row, gr->du, status);
  MOE_TRY(launched());
  // --- data gradients (FP8 GEMMs on the transposed weights)
  void* dh = at<void>(ws, B.dh);
  void* dab = at<void>(ws, B.dab);
  void* dx = at<void>(ws, B.dx);
  MOE_TRY(quant_rows(dy, R, static_cast<int>(D), at<void>(ws, B.dyq), at<void>(ws, B.dys), R, pow2, st));
  MOE_TRY(fp8gemm_bf16(wt->w2t, wt->w2t_scale, E * I, static_cast<int>(I), static_cast<int>(D), at<void>(ws, B.dyq),
                       at<float>(ws, B.dys), R, R, dh, I, Ei, groups, mt_total, cgroup, R, 0, 0, queue + 2, status, st));
  swiglu_bwd_kernel<<<ew_blocks(R * I / 8), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(ab),
                                                           static_cast<const __nv_bfloat16*>(dh), R,
                                                           static_cast<int>(I), static_cast<__nv_bfloat16*>(dab));
  MOE_TRY(launched());
  MOE_TRY(quant_rows(dab, R, static_cast<int>(I2), at<void>(ws, B.dabq), at<void>(ws, B.dabs), R, pow2, st));
  MOE_TRY(fp8gemm_bf16(wt->w13t, wt->w13t_scale, E * D, static_cast<int>(D), static_cast<int>(I2),
                       at<void>(ws, B.dabq), at<float>(ws, B.dabs), R, R, dx, D, Ei, groups, mt_total, cgroup, R, 0,
                       0, queue + 3, status, st));
  // --- shared experts: every token, output gradient G itself
  void* ab_s = at<void>(ws, B.ab_s);
  void* hsb = at<void>(ws, B.hsb);
  void* dh_s = at<void>(ws, B.dh_s);
  void* dab_s = at<void>(ws, B.dab_s);
  void* dx_s = at<void>(ws, B.dx_s);
  if (Ns > 0) {
    MOE_TRY(fp8gemm_bf16(w->ws13, w->ws13_scale, Ns * I2, static_cast<int>(I2), static_cast<int>(D), uq, uqs, T, T,
                         ab_s, I2, Nsi, nullptr, nullptr, nullptr, 0, Ti, 0, queue + 4, status, st));
    swiglu_fwd_kernel<<<ew_blocks(Ns * T * I / 8), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(ab_s), Ns * T,
                                                                  static_cast<int>(I), static_cast<__nv_bfloat16*>(hsb));
    MOE_TRY(launched());
    MOE_TRY(quant_rows(dout, T, static_cast<int>(D), at<void>(ws, B.Gq), at<void>(ws, B.Gs), T, pow2, st));
    MOE_TRY(fp8gemm_bf16(wt->ws2t, wt->ws2t_scale, Ns * I, static_cast<int>(I), static_cast<int>(D),
                         at<void>(ws, B.Gq), at<float>(ws, B.Gs), T, T, dh_s, I, Nsi, nullptr, nullptr, nullptr, 0, Ti,
                         0, queue + 5, status, st));
    swiglu_bwd_kernel<<<ew_blocks(Ns * T * I / 8), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(ab_s),
                                                                  static_cast<const __nv_bfloat16*>(dh_s), Ns * T,
                                                                  static_cast<int>(I),
                                                                  static_cast<__nv_bfloat16*>(dab_s));
    MOE_TRY(launched());
    MOE_TRY(quant_rows(dab_s, Ns * T, static_cast<int>(I2), at<void>(ws, B.dabsq), at<void>(ws, B.dabss), Ns * T,
                       pow2, st));
    MOE_TRY(fp8gemm_bf16(wt->ws13t, wt->ws13t_scale, Ns * D, static_cast<int>(D), static_cast<int>(I2),
                         at<void>(ws, B.dabsq), at<float>(ws, B.dabss), Ns * T, Ns * T, dx_s, D, Nsi, nullptr,
                         nullptr, nullptr, 0, Ti, Ti, queue + 6, status, st));
  }
  gather_dx_kernel<<<static_cast<unsigned>(T), 128, 0, st>>>(static_cast<const __nv_bfloat16*>(dx), slot, d.k, R,
                                                              static_cast<const __nv_bfloat16*>(dx_s), Nsi, Ti,
                                                              static_cast<int>(D), gr->du);
  MOE_TRY(launched());
  dcent_kernel<<<dim3(static_cast<unsigned>(E), static_cast<unsigned>(cdiv(D, 256))), 256, 0, st>>>(
      dz_row, perm, offsets, reinterpret_cast<const __nv_bfloat16*>(u), static_cast<int>(D), gr->dcentroids);
  MOE_TRY(launched());
  // --- weight gradients: operands quantised along the tokens (128-token
  // blocks from each expert's first token), products on the bf16 path
  int32_t* pad_off = at<int32_t>(ws, B.pad_off);
  int32_t* row_of_col = at<int32_t>(ws, B.row_of_col);
  WgradGroup* wg_r = at<WgradGroup>(ws, B.wg_r);
  pad_plan_kernel<<<1, 1024, 0, st>>>(offsets, Ei, static_cast<int>(B.Rp), 128, pad_off, row_of_col, status);
  MOE_TRY(launched());
  wgrad_table_kernel<<<static_cast<unsigned>(cdiv(E, 256)), 256, 0, st>>>(pad_off, Ei, wg_r);
  MOE_TRY(launched());
  void* xT = at<void>(ws, B.xT);
  void* dyT = at<void>(ws, B.dyT);
  void* hT = at<void>(ws, B.hT);
  void* dabT = at<void>(ws, B.dabT);
  const int32_t* live = pad_off + Ei;  // padded total: the columns the weight-gradient GEMM reads
  MOE_TRY(transpose_fq(u, Ti, static_cast<int>(D), 0, row_of_col, perm, live, B.Rp, xT, B.Rp, 0, 1, pow2, st));
  MOE_TRY(transpose_fq(dy, static_cast<int>(R), static_cast<int>(D), 0, row_of_col, nullptr, live, B.Rp, dyT, B.Rp,
                       0, 1, pow2, st));
  MOE_TRY(transpose_fq(hb, static_cast<int>(R), static_cast<int>(I), 0, row_of_col, nullptr, live, B.Rp, hT, B.Rp, 0, 1,
                       pow2, st));
  MOE_TRY(transpose_fq(dab, static_cast<int>(R), static_cast<int>(I2), 0, row_of_col, nullptr, live, B.Rp, dabT,
                       B.Rp, 0, 1, pow2, st));
  MOE_TRY(wgrad(dyT, B.Rp, static_cast<int>(D), hT, B.Rp, static_cast<int>(I), wg_r, Ei, gr->dw2, queue + 8, status,
                st));
  MOE_TRY(wgrad(dabT, B.Rp, static_cast<int>(I2), xT, B.Rp, static_cast<int>(D), wg_r, Ei, gr->dw13, queue + 9,
                status, st));
  if (Ns > 0) {
    void* uT = at<void>(ws, B.uT);
    void* GT = at<void>(ws, B.GT);
    void* hsT = at<void>(ws, B.hsT);
    void* dabsT = at<void>(ws, B.dabsT);
    const int Tp = static_cast<int>(B.Tp);
    MOE_TRY(transpose_fq(u, Ti, static_cast<int>(D), 0, nullptr, nullptr, nullptr, Tp, uT, Tp, 0, 1, pow2, st));
    MOE_TRY(transpose_fq(dout, Ti, static_cast<int>(D), 0, nullptr, nullptr, nullptr, Tp, GT, Tp, 0, 1, pow2, st));
    MOE_TRY(transpose_fq(hsb, Ti, static_cast<int>(I), T * I, nullptr, nullptr, nullptr, Tp, hsT, Ns * Tp, Tp, Nsi,
                         pow2, st));
    MOE_TRY(transpose_fq(dab_s, Ti, static_cast<int>(I2), T * I2, nullptr, nullptr, nullptr, Tp, dabsT, Ns * Tp, Tp,
                         Nsi, pow2, st));
    WgradGroup* wg_s2 = at<WgradGroup>(ws, B.wg_s2);
    WgradGroup* wg_s13 = at<WgradGroup>(ws, B.wg_s13);
    wgrad_strided_table_kernel<<<1, 256, 0, st>>>(Nsi, 0, Tp, Tp, wg_s2);   // A = G^T, B = h_s^T
    MOE_TRY(launched());
    wgrad_strided_table_kernel<<<1, 256, 0, st>>>(Nsi, Tp, 0, Tp, wg_s13);  // A = dab_s^T, B = u^T
    MOE_TRY(launched());
    MOE_TRY(wgrad(GT, Tp, static_cast<int>(D), hsT, Ns * Tp, static_cast<int>(I), wg_s2, Nsi, gr->dws2, queue + 10,
                  status, st));
    MOE_TRY(wgrad(dabsT, Ns * Tp, static_cast<int>(I2), uT, Tp, static_cast<int>(D), wg_s13, Nsi, gr->dws13,
                  queue + 11, status, st));
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_forward_profiled(const moe_dims* dims, const moe_weights* w, const uint16_t* u, const float* bias,
                                uint16_t* out, int32_t* counts_out, void* ws, size_t ws_bytes, void* stream,
                                void* const* events, int32_t n_events) {
  return forward_impl(dims, w, u, bias, out, counts_out, ws, ws_bytes, stream, events, n_events, nullptr);
}

moe_status moe_plan_replicas(int32_t E, const int32_t* counts, int32_t n_extra, int32_t* replica_first,
                             int32_t* replica_count, int32_t* slot_expert) {
  if (E <= 0 || E > 1024 || n_extra < 0 || n_extra > 1024 || !counts || !replica_first || !replica_count ||
      (!slot_expert && E + n_extra > 0))
    return MOE_ERR_INVALID_ARG;
  for (int e = 0; e < E; ++e) {
    if (counts[e] < 0) return MOE_ERR_INVALID_ARG;
    replica_count[e] = 1;
  }
  // each extra copy goes to the expert with the highest load per copy
  // (counts[e] / copies[e], compared exactly as counts[a] * copies[b] vs
  // counts[b] * copies[a]; ties to the lower index)
  for (int r = 0; r < n_extra; ++r) {
    int best = 0;
    for (int e = 1; e < E; ++e)
      if (int64_t(counts[e]) * replica_count[best] > int64_t(counts[best]) * replica_count[e]) best = e;
    ++replica_count[best];
  }
  int32_t p = 0;
  for (int e = 0; e < E; ++e) {
    replica_first[e] = p;
    for (int c = 0; c < replica_count[e]; ++c) slot_expert[p++] = e;
  }
  return MOE_OK;
}

moe_status moe_forward_replicated(const moe_dims* dims, const moe_weights* w, const uint16_t* u, const float* bias,
                                  const int32_t* replica_first, const int32_t* replica_count,
                                  const int32_t* slot_expert, int32_t n_slots, uint16_t* out, int32_t* counts_out,
                                  void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_dims(dims));
  if (!replica_first || !replica_count || !slot_expert || n_slots < dims->E || n_slots > 2048)
    return MOE_ERR_INVALID_ARG;
  const ReplicaPlan rp{replica_first, replica_count, slot_expert, n_slots};
  return forward_impl(dims, w, u, bias, out, counts_out, ws, ws_bytes, stream, nullptr, 0, &rp);
}

moe_status moe_backward_workspace_size(const moe_dims* dims, size_t* bytes) {
  MOE_TRY(check_dims(dims));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_bwd_layout(*dims).total;
  return MOE_OK;
}

moe_status moe_transpose_expert_weights(int32_t n_experts, int32_t inter, int32_t d, const uint16_t* w13,
                                        const uint16_t* w2, uint16_t* w13t, uint16_t* w2t, void* stream) {
  if (n_experts <= 0 || n_experts > 65535 || inter <= 0 || d <= 0 || inter % 128 || d % 128) return MOE_ERR_INVALID_ARG;
  if (!w13 || !w2 || !w13t || !w2t) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t I2 = 2 * int64_t(inter);
  MOE_TRY(
      transpose_bf16(w13, static_cast<int>(I2), d, I2 * d, nullptr, nullptr, I2, w13t, I2, I2 * d, n_experts, st));
  return transpose_bf16(w2, d, inter, int64_t(d) * inter, nullptr, nullptr, d, w2t, d, int64_t(d) * inter, n_experts, st);
}

moe_status moe_transpose_expert_weights_fp8(int32_t n_experts, int32_t inter, int32_t d, const uint8_t* w13,
                                            const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                            uint8_t* w13t, float* w13t_scale, uint8_t* w2t, float* w2t_scale,
                                            void* stream) {
  if (n_experts <= 0 || n_experts > 65535 || inter <= 0 || d <= 0 || inter % 128 || d % 128) return MOE_ERR_INVALID_ARG;
  if (!w13 || !w2 || !w13t || !w2t || !w13_scale || !w2_scale || !w13t_scale || !w2t_scale)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(w13) || !aligned16(w2) || !aligned16(w13t) || !aligned16(w2t)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int I2 = 2 * inter;
  transpose_u8_kernel<<<dim3(static_cast<unsigned>(d / 64), static_cast<unsigned>(I2 / 64),
                             static_cast<unsigned>(n_experts)), 256, 0, st>>>(w13, I2, d, int64_t(I2) * d, w13t);
  MOE_TRY(launched());
  transpose_u8_kernel<<<dim3(static_cast<unsigned>(inter / 64), static_cast<unsigned>(d / 64),
                             static_cast<unsigned>(n_experts)), 256, 0, st>>>(w2, d, inter, int64_t(d) * inter, w2t);
  MOE_TRY(launched());
  transpose_f32_kernel<<<ew_blocks(int64_t(n_experts) * (I2 / 128) * (d / 128)), 256, 0, st>>>(
      w13_scale, I2 / 128, d / 128, n_experts, w13t_scale);
  MOE_TRY(launched());
  transpose_f32_kernel<<<ew_blocks(int64_t(n_experts) * (d / 128) * (inter / 128)), 256, 0, st>>>(
      w2_scale, d / 128, inter / 128, n_experts, w2t_scale);
  return launched();
}

moe_status moe_backward(const moe_dims* dims, const moe_weights* w, const moe_weights_t* wt, const uint16_t* u,
                        const float* bias, const uint16_t* dout, const moe_grads* gr, void* ws, size_t ws_bytes,
                        void* stream) {
  MOE_TRY(check_dims(dims));
  MOE_TRY(check_weights(*dims, w));
  const moe_dims& d = *dims;
  if (!wt || !wt->w13t || !wt->w2t || (d.n_shared > 0 && (!wt->ws13t || !wt->ws2t))) return MOE_ERR_INVALID_ARG;
  if (is_fp8(d) && (!wt->w13t_scale || !wt->w2t_scale || (d.n_shared > 0 && (!wt->ws13t_scale || !wt->ws2t_scale))))
    return MOE_ERR_INVALID_ARG;
  if (!gr || (d.T > 0 && !gr->du) || !gr->dcentroids || !gr->dw13 || !gr->dw2 ||
      (d.n_shared > 0 && (!gr->dws13 || !gr->dws2)))
    return MOE_ERR_INVALID_ARG;
  // vector stores of du, TMA stores of the weight gradients
  if (!aligned16(gr->du) || !aligned16(gr->dw13) || !aligned16(gr->dw2) ||
      (d.n_shared > 0 && (!aligned16(gr->dws13) || !aligned16(gr->dws2))))
    return MOE_ERR_INVALID_ARG;
  if (!bias || (d.T > 0 && (!u || !dout)) || !aligned16(u) || !aligned16(dout)) return MOE_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return MOE_ERR_INVALID_ARG;
  const BwdLayout B = make_bwd_layout(d);
  if (ws_bytes < B.total) return MOE_ERR_WORKSPACE;
  const Layout& L = B.f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t T = d.T, R = T * d.k, E = d.E, I = d.inter, D = d.d, Ns = d.n_shared, I2 = 2 * I;
  int* status = at<int>(ws, L.status);
  int* queue = at<int>(ws, B.queue);
  MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, sizeof(int), st)));
  MOE_TRY(cuda_ok(cudaMemsetAsync(queue, 0, 16 * sizeof(int), st)));
  if (T == 0) {  // no tokens: zero gradients
    MOE_TRY(cuda_ok(cudaMemsetAsync(gr->dcentroids, 0, E * D * 4, st)));
    MOE_TRY(cuda_ok(cudaMemsetAsync(gr->dw13, 0, E * I2 * D * 4, st)));
    MOE_TRY(cuda_ok(cudaMemsetAsync(gr->dw2, 0, E * D * I * 4, st)));
    if (Ns > 0) {
      MOE_TRY(cuda_ok(cudaMemsetAsync(gr->dws13, 0, Ns * I2 * D * 4, st)));
      MOE_TRY(cuda_ok(cudaMemsetAsync(gr->dws2, 0, Ns * D * I * 4, st)));
    }
    return MOE_OK;
  }
  const int W = static_cast<int>((T + 31) / 32);
  uint32_t* mask = at<uint32_t>(ws, L.mask);
  MOE_TRY(cuda_ok(cudaMemsetAsync(mask, 0, sizeof(uint32_t) * size_t(E) * W, st)));
  // --- the forward's routing and dispatch, recomputed
  int32_t* idx = at<int32_t>(ws, L.idx);
  float* gate = at<float>(ws, L.gate);
  float* z = at<float>(ws, L.z);
  MOE_TRY(enqueue_route(d, u, w->centroids, bias, idx, gate, at<int32_t>(ws, L.counts), mask, z, status, st));
  if (is_fp8(d)) return backward_fp8(d, B, w, wt, u, dout, gr, ws, st);
  GroupEntry* groups = at<GroupEntry>(ws, L.groups);
  int32_t* mt_total = at<int32_t>(ws, L.mt_total);
  int32_t* cgroup = at<int32_t>(ws, L.cgroup);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* perm = at<int32_t>(ws, L.perm);
  int32_t* slot = at<int32_t>(ws, L.slot);
  void* x = at<void>(ws, L.x);
  MOE_TRY(enqueue_dispatch(d, idx, u, mask, at<int32_t>(ws, L.wprefix), at<int32_t>(ws, L.cnt), offsets, groups,
                           mt_total, cgroup, perm, slot, x, nullptr, nullptr, nullptr, status, st));
  const int64_t chunks = cdiv(R + int64_t(kChunkBf16 - 1) * E, kChunkBf16);
  // kernel shapes (XShape) of the backward's GEMMs, measured at V3 size
  constexpr bool kWideAB = false, kWideDh = false, kWideDx = false, kWideShared = true;
  void* ab = at<void>(ws, B.ab);
  void* h = at<void>(ws, L.h);
  void* y = at<void>(ws, L.y);
  // --- routed experts: a, b (gate/up pre-activations), h.  The experts'
  // outputs y are not recomputed: the gates' gradient G . y is (dh . h) / g
  // (gate_grad_kernel), from dh below.
  MOE_TRY(xgemm_bf16(w->w13, E * I2, static_cast<int>(I2), static_cast<int>(D), x, R, ab, I2, static_cast<int>(E),
                     groups, mt_total, cgroup, chunks, 0, 0, queue + 0, status, kWideAB, st));
  swiglu_fwd_kernel<<<ew_blocks(R * I / 8), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(ab), R, static_cast<int>(I),
                                                       static_cast<__nv_bfloat16*>(h));
  MOE_TRY(launched());
  // --- the routed rows' output gradient dy = g G, then dh = dy W2
  void* dy = at<void>(ws, B.dy);
  float* dz_row = at<float>(ws, B.dz_row);
  scale_rows_kernel<<<static_cast<unsigned>(T), 128, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(dout), slot, gate,
                                                              d.k, static_cast<int>(D), R,
                                                              static_cast<__nv_bfloat16*>(dy));
  MOE_TRY(launched());
  void* dh = at<void>(ws, B.dh);
  void* dab = at<void>(ws, B.dab);
  void* dx = at<void>(ws, B.dx);
  MOE_TRY(xgemm_bf16(wt->w2t, E * I, static_cast<int>(I), static_cast<int>(D), dy, R, dh, I, static_cast<int>(E), groups,
                     mt_total, cgroup, chunks, 0, 0, queue + 2, status, kWideDh, st));
  // --- gates backward: dz, du = G + router share
  const LogitsSplit sp = logits_split(d);
  gate_grad_kernel<<<static_cast<unsigned>(T), 128, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(dout), static_cast<const __nv_bfloat16*>(dh),
      static_cast<const __nv_bfloat16*>(h), static_cast<int>(I), slot, idx, gate, z, sp.splits, T * E,
      reinterpret_cast<const __nv_bfloat16*>(w->centroids), static_cast<int>(D), d.k, static_cast<int>(E), R, dz_row,
      gr->du, status);
  MOE_TRY(launched());
  swiglu_bwd_kernel<<<ew_blocks(R * I / 8), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(ab),
                                                       static_cast<const __nv_bfloat16*>(dh), R, static_cast<int>(I),
                                                       static_cast<__nv_bfloat16*>(dab));
  MOE_TRY(launched());
  MOE_TRY(xgemm_bf16(wt->w13t, E * D, static_cast<int>(D), static_cast<int>(I2), dab, R, dx, D, static_cast<int>(E),
                     groups, mt_total, cgroup, chunks, 0, 0, queue + 3, status, kWideDx, st));
  // --- shared experts: every token, the output gradient is G itself
  void* ab_s = at<void>(ws, B.ab_s);
  void* h_s = at<void>(ws, L.hsh);
  void* dh_s = at<void>(ws, B.dh_s);
  void* dab_s = at<void>(ws, B.dab_s);
  void* dx_s = at<void>(ws, B.dx_s);
  if (Ns > 0) {
    const int Ti = static_cast<int>(T), Nsi = static_cast<int>(Ns);
    MOE_TRY(xgemm_bf16(w->ws13, Ns * I2, static_cast<int>(I2), static_cast<int>(D), u, T, ab_s, I2, Nsi, nullptr,
                       nullptr, nullptr, 0, Ti, 0, queue + 4, status, kWideShared, st));
    swiglu_fwd_kernel<<<ew_blocks(Ns * T * I / 8), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(ab_s), Ns * T,
                                                              static_cast<int>(I), static_cast<__nv_bfloat16*>(h_s));
    MOE_TRY(launched());
    MOE_TRY(xgemm_bf16(wt->ws2t, Ns * I, static_cast<int>(I), static_cast<int>(D), dout, T, dh_s, I, Nsi, nullptr,
                       nullptr, nullptr, 0, Ti, 0, queue + 5, status, kWideShared, st));
    swiglu_bwd_kernel<<<ew_blocks(Ns * T * I / 8), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(ab_s),
                                                              static_cast<const __nv_bfloat16*>(dh_s), Ns * T,
                                                              static_cast<int>(I), static_cast<__nv_bfloat16*>(dab_s));
    MOE_TRY(launched());
    MOE_TRY(xgemm_bf16(wt->ws13t, Ns * D, static_cast<int>(D), static_cast<int>(I2), dab_s, Ns * T, dx_s, D, Nsi,
                       nullptr, nullptr, nullptr, 0, Ti, Ti, queue + 6, status, kWideShared, st));
  }
  gather_dx_kernel<<<static_cast<unsigned>(T), 128, 0, st>>>(static_cast<const __nv_bfloat16*>(dx), slot, d.k, R,
                                                              static_cast<const __nv_bfloat16*>(dx_s),
                                                              static_cast<int>(Ns), static_cast<int>(T),
                                                              static_cast<int>(D), gr->du);
  MOE_TRY(launched());
  // --- centroid gradient
  dcent_kernel<<<dim3(static_cast<unsigned>(E), static_cast<unsigned>(cdiv(D, 256))), 256, 0, st>>>(
      dz_row, perm, offsets, reinterpret_cast<const __nv_bfloat16*>(u), static_cast<int>(D), gr->dcentroids);
  MOE_TRY(launched());
  // --- weight gradients of the routed experts: the expert's tokens along K
  int32_t* pad_off = at<int32_t>(ws, B.pad_off);
  int32_t* row_of_col = at<int32_t>(ws, B.row_of_col);
  WgradGroup* wg_r = at<WgradGroup>(ws, B.wg_r);
  pad_plan_kernel<<<1, 1024, 0, st>>>(offsets, static_cast<int>(E), static_cast<int>(B.Rp), 64, pad_off, row_of_col,
                                      status);
  MOE_TRY(launched());
  wgrad_table_kernel<<<static_cast<unsigned>(cdiv(E, 256)), 256, 0, st>>>(pad_off, static_cast<int>(E), wg_r);
  MOE_TRY(launched());
  void* xT = at<void>(ws, B.xT);
  void* dyT = at<void>(ws, B.dyT);
  void* hT = at<void>(ws, B.hT);
  void* dabT = at<void>(ws, B.dabT);
  // the padding columns are written as zeros by the transposes themselves
  const int32_t* live = pad_off + E;  // padded total: the columns the weight-gradient GEMM reads
  MOE_TRY(transpose_bf16(x, static_cast<int>(R), static_cast<int>(D), 0, row_of_col, live, B.Rp, xT, B.Rp, 0, 1, st));
  MOE_TRY(transpose_bf16(dy, static_cast<int>(R), static_cast<int>(D), 0, row_of_col, live, B.Rp, dyT, B.Rp, 0, 1, st));
  MOE_TRY(transpose_bf16(h, static_cast<int>(R), static_cast<int>(I), 0, row_of_col, live, B.Rp, hT, B.Rp, 0, 1, st));
  MOE_TRY(
      transpose_bf16(dab, static_cast<int>(R), static_cast<int>(I2), 0, row_of_col, live, B.Rp, dabT, B.Rp, 0, 1, st));
  MOE_TRY(wgrad(dyT, B.Rp, static_cast<int>(D), hT, B.Rp, static_cast<int>(I), wg_r, static_cast<int>(E), gr->dw2,
                queue + 8, status, st));
  MOE_TRY(wgrad(dabT, B.Rp, static_cast<int>(I2), xT, B.Rp, static_cast<int>(D), wg_r, static_cast<int>(E), gr->dw13,
                queue + 9, status, st));
  // --- weight gradients of the shared experts (K = all tokens, padded)
  if (Ns > 0) {
    void* uT = at<void>(ws, B.uT);
    void* GT = at<void>(ws, B.GT);
    void* hsT = at<void>(ws, B.hsT);
    void* dabsT = at<void>(ws, B.dabsT);
    const int Tp = static_cast<int>(B.Tp), Ti = static_cast<int>(T), Nsi = static_cast<int>(Ns);
    MOE_TRY(transpose_bf16(u, Ti, static_cast<int>(D), 0, nullptr, nullptr, Tp, uT, Tp, 0, 1, st));
    MOE_TRY(transpose_bf16(dout, Ti, static_cast<int>(D), 0, nullptr, nullptr, Tp, GT, Tp, 0, 1, st));
    MOE_TRY(transpose_bf16(h_s, Ti, static_cast<int>(I), T * I, nullptr, nullptr, Tp, hsT, Ns * Tp, Tp, Nsi, st));
    MOE_TRY(transpose_bf16(dab_s, Ti, static_cast<int>(I2), T * I2, nullptr, nullptr, Tp, dabsT, Ns * Tp, Tp, Nsi, st));
    WgradGroup* wg_s2 = at<WgradGroup>(ws, B.wg_s2);
    WgradGroup* wg_s13 = at<WgradGroup>(ws, B.wg_s13);
    wgrad_strided_table_kernel<<<1, 256, 0, st>>>(Nsi, 0, Tp, Tp, wg_s2);       // A = G^T, B = h_s^T
    MOE_TRY(launched());
    wgrad_strided_table_kernel<<<1, 256, 0, st>>>(Nsi, Tp, 0, Tp, wg_s13);      // A = dab_s^T, B = u^T
    MOE_TRY(launched());
    MOE_TRY(wgrad(GT, Tp, static_cast<int>(D), hsT, Ns * Tp, static_cast<int>(I), wg_s2, Nsi, gr->dws2, queue + 10,
                  status, st));
    MOE_TRY(wgrad(dabsT, Ns * Tp, static_cast<int>(I2), uT, Tp, static_cast<int>(D), wg_s13, Nsi, gr->dws13, queue + 11,
                  status, st));
  }
  return MOE_OK;
}

moe_status moe_pack_gate_up(const uint16_t* w1, const uint16_t* w3, int32_t E, int32_t inter, int32_t d,
                            uint16_t* w13, void* stream) {
  if (!w1 || !w3 || !w13 || E <= 0 || inter <= 0 || d <= 0 || inter % 128 || d % 8) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w1) || !aligned16(w3) || !aligned16(w13)) return MOE_ERR_INVALID_ARG;
  pack_gate_up_kernel<<<148 * 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(w1), reinterpret_cast<const uint4*>(w3), E, inter, d,
      reinterpret_cast<uint4*>(w13));
  return launched();
}

moe_status moe_quantize_fp8_blocks(const uint16_t* w, int64_t rows, int32_t cols, uint8_t* q, float* scale,
                                   int32_t pow2_scales, void* stream) {
  if (!w || !q || !scale || rows <= 0 || cols <= 0 || rows % 128 || cols % 128) return MOE_ERR_INVALID_ARG;
  if (rows / 128 > 65535 * 64) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(w) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // grid.y is limited to 65535 block rows: split taller matrices
  for (int64_t r0 = 0; r0 < rows; r0 += int64_t(65535) * 128) {
    const int64_t r = rows - r0 < int64_t(65535) * 128 ? rows - r0 : int64_t(65535) * 128;
    dim3 grid(cols / 128, static_cast<unsigned>(r / 128));
    quantize_blocks_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(w) + r0 * cols, cols,
                                                 q + r0 * cols, scale + (r0 / 128) * (cols / 128), pow2_scales != 0);
    MOE_TRY(launched());
  }
  return MOE_OK;
}

moe_status moe_read_device_status(const void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status>(v);
}

moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int32_t timeout_us, void* stream) {
  if (!ws || ws_bytes < 256 || timeout_us <= 0 || timeout_us > 10000000) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_TRY(cuda_ok(cudaMemsetAsync(ws, 0, sizeof(int), st)));
  selftest_timeout_kernel<<<1, 32, 0, st>>>(static_cast<int*>(ws), uint64_t(timeout_us) * 1000ull);
  return launched();
}

}  // extern "C"

// =================================================================== route without a workspace
// moe_route_noalloc: the router for callers that cannot allocate device memory.
// Its only scratch, the [T, E] fp32 logits, is this fixed array; the runtime
// creates it on every device that loads the library.  Host code must not pass
// the symbol itself to a kernel (on the host it names a stand-in, not device
// memory): the address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) float route_logits_scratch[MOE_ROUTE_NOALLOC_MAX_LOGITS];

namespace {

constexpr int kMaxDevices = 64;
std::mutex scratch_mutex;
struct ScratchCache {
  unsigned long long ctx_id;  // unique id of the context the address belongs to (0: none yet)
  float* addr;
};
ScratchCache scratch_cache[kMaxDevices] = {};

// Driver calls that identify the current context; every context of the
// process has its own id, never reused, so a device reset (a new primary
// context, whose copy of the array may sit elsewhere) is always noticed.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <class F>
F driver_fn(const char* name, int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(p);
}

moe_status current_ctx_id(unsigned long long* id) {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 12000);
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
  if (!get_current || !get_id) return MOE_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  *id = 0;
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  return MOE_OK;
}

// Device address of route_logits_scratch in the current device's current
// context: looked up with cudaGetSymbolAddress the first time (which also
// makes the device's primary context current if it was not) and cached per
// device together with the context's id; looked up again whenever the
// context has changed since (for instance after cudaDeviceReset).
moe_status route_scratch(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(scratch_mutex);
  unsigned long long id = 0;
  MOE_TRY(current_ctx_id(&id));
  ScratchCache& c = scratch_cache[dev];
  if (id == 0 || c.ctx_id != id || !c.addr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, route_logits_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    MOE_TRY(current_ctx_id(&id));
    if (id == 0) return MOE_ERR_CUDA;
    c.ctx_id = id;
    c.addr = static_cast<float*>(p);
  }
  *out = c.addr;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_route_noalloc(const moe_dims* dims, const uint16_t* u, const uint16_t* centroids,
                                        const float* bias, int32_t* topk_idx, float* topk_gate, int32_t* counts,
                                        int32_t* device_status, void* stream) {
  MOE_TRY(check_dims(dims));
  // token-sized buffers may be empty (null) when T == 0
  const bool empty = dims->T == 0;
  if (!centroids || !bias || !counts || (!empty && (!u || !topk_idx || !topk_gate))) return MOE_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(centroids)) return MOE_ERR_INVALID_ARG;
  if (int64_t(dims->T) * dims->E > MOE_ROUTE_NOALLOC_MAX_LOGITS) return MOE_ERR_UNSUPPORTED;
  float* z = nullptr;
  MOE_TRY(route_scratch(&z));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (device_status) MOE_TRY(cuda_ok(cudaMemsetAsync(device_status, 0, sizeof(int32_t), st)));
  if (dims->T == 0) return cuda_ok(cudaMemsetAsync(counts, 0, sizeof(int32_t) * dims->E, st));
  return enqueue_route(*dims, u, centroids, bias, topk_idx, topk_gate, counts, nullptr, z, device_status, st);
}
