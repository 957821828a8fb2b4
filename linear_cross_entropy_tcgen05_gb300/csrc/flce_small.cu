// flce_small.cu -- the bandwidth/latency-bound helper kernels of fused linear
// cross-entropy: the forward finalize (combine the vocabulary splits into lse, form the
// row losses, reduce them in a fixed order), the backward prep (valid-row count and
// per-row gradient coefficients), the valid-row compaction (row list and gather, for both
// passes; the scatter back of dX), the fp32 -> bf16 cast of dX, and the launch counter and
// GEMM timing diagnostics.
#include <atomic>
#include <mutex>
#include <vector>

#include <cuda_bf16.h>
#include <math_constants.h>

#include "flce_internal.h"
#include "sm103_ptx.cuh"
#include "vec_split.h"

namespace flce {

namespace {
constexpr float kLog2e = 1.4426950408889634f;
}

// ---------------------------------------------------------------------------------
// ---------------------------------------------------------------------------------

// A GEMM whose pipeline wait ran out has set FLCE_DEVERR_TIMEOUT in this call's error word
// (cleared when the call began) and left its outputs (the forward's partial statistics, a
// part of the dX accumulator) unwritten; they may hold a previous call's values, so the
// kernels that read them write NaN instead.
__device__ __forceinline__ bool call_timed_out(const int* err) {
  return err != nullptr && (*reinterpret_cast<const volatile int*>(err) & FLCE_DEVERR_TIMEOUT) != 0;
}

// Combine each row's partial statistics into lse and the row loss (FIN_LOSS), into one
// vocabulary shard's statistics (FIN_SHARD_STATS), or combine K shards' statistics
// (FIN_COMBINE); then reduce the loss deterministically (per-block fp64 partial sums,
// then one block). After a timeout every result of the call is NaN.
__global__ void __launch_bounds__(kFinalizeThreads)
    flce_finalize_rows_kernel(const FinalizeParams p) {
  const int row = int(blockIdx.x) * kFinalizeThreads + int(threadIdx.x);
  const bool timed_out = call_timed_out(p.err);
  double contrib = 0.0, den = 0.0;
  int valid = 0, correct = 0;
  if (row < p.N) {
    float M = -CUDART_INF_F, d = 0.f, sz = 0.f, zy = 0.f;
    int owners = 0, best_idx = 0;
    if (p.mode == FIN_COMBINE) {
      for (int s = 0; s < p.S; ++s) M = fmaxf(M, p.stats[(size_t(s) * 4 + 0) * p.N + row]);
      for (int s = 0; s < p.S; ++s) {
        const float* st = p.stats + size_t(s) * 4 * p.N;
        d += exp2f((st[row] - M) * kLog2e);
        sz += st[size_t(p.N) + row];
        zy += st[2 * size_t(p.N) + row];
        owners += st[3 * size_t(p.N) + row] != 0.f ? 1 : 0;
      }
    } else if (p.slot != nullptr && p.slot[row] < 0) {
      // an ignored row of a forward that ran on the valid rows only: no statistics
    } else {
      const int prow = p.slot != nullptr ? p.slot[row] : row;  // where this row's partials sit
      float best = -CUDART_INF_F;
      for (int s = 0; s < p.S; ++s) {
        const float m = p.part_m[size_t(s) * p.N + prow];
        M = fmaxf(M, m);
        if (p.part_idx != nullptr) {
          const int idx = p.part_idx[size_t(s) * p.N + prow];
          if (m > best || (m == best && idx < best_idx)) {
            best = m;
            best_idx = idx;
          }
        }
      }
      for (int s = 0; s < p.S; ++s) {
        const size_t o = size_t(s) * p.N + prow;
        d += p.part_d[o] * exp2f((p.part_m[o] - M) * kLog2e);
        sz += p.part_s[o];
      }
      zy = p.tgt[prow];
    }
    const int y = p.targets[row];
    // the lse of an ignored row is 0 (the loss needs none; a forward that runs on the
    // valid rows only does not compute it)
    float lse = y == p.ignore_index && p.mode != FIN_SHARD_STATS ? 0.f : M + logf(d);
    if (timed_out) lse = CUDART_NAN_F;
    if (p.mode == FIN_SHARD_STATS) {
      const int rel = y - p.v_offset;
      const bool own = y != p.ignore_index && rel >= 0 && rel < p.V_local;
      p.stats_out[row] = lse;
      p.stats_out[size_t(p.N) + row] = timed_out ? CUDART_NAN_F : sz;
      p.stats_out[2 * size_t(p.N) + row] = timed_out ? CUDART_NAN_F : (own ? zy : 0.f);
      p.stats_out[3 * size_t(p.N) + row] = own ? 1.f : 0.f;
      return;
    }
    p.lse[row] = lse;
    if (p.predicted != nullptr) p.predicted[row] = best_idx;
    float ell = 0.f;
    if (y != p.ignore_index) {
      valid = 1;
      const bool bad = y < 0 || y >= p.V || (p.mode == FIN_COMBINE && owners != 1);
      if (bad) {
        atomicOr(p.err, FLCE_DEVERR_BAD_TARGET);
        ell = CUDART_NAN_F;
        den = 1.0;
      } else {
        const float wy = p.cw != nullptr ? p.cw[y] : 1.f;
        const float wtot = p.cw != nullptr ? *p.wtot : float(p.V);
        ell = (1.f - p.eps) * wy * (lse - zy) + p.zscale * lse * lse;
        if (p.eps != 0.f) ell += p.eps / float(p.V) * (wtot * lse - sz);
        den = double(wy);
        correct = (p.predicted != nullptr && best_idx == y) ? 1 : 0;
      }
    }
    if (timed_out) ell = CUDART_NAN_F;
    if (p.reduction == 2) p.loss[row] = ell;
    contrib = double(ell);
  }
  if (p.mode == FIN_SHARD_STATS) return;
  // fixed-order block reduction
  __shared__ double ssum[kFinalizeThreads];
  __shared__ double sden[kFinalizeThreads];
  __shared__ int scnt[kFinalizeThreads];
  __shared__ int scor[kFinalizeThreads];
  ssum[threadIdx.x] = contrib;
  sden[threadIdx.x] = den;
  scnt[threadIdx.x] = valid;
  scor[threadIdx.x] = correct;
  __syncthreads();
  for (int o = kFinalizeThreads / 2; o > 0; o >>= 1) {
    if (int(threadIdx.x) < o) {
      ssum[threadIdx.x] += ssum[threadIdx.x + o];
      sden[threadIdx.x] += sden[threadIdx.x + o];
      scnt[threadIdx.x] += scnt[threadIdx.x + o];
      scor[threadIdx.x] += scor[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.block_sum[blockIdx.x] = ssum[0];
    p.block_wsum[blockIdx.x] = sden[0];
    p.block_cnt[blockIdx.x] = scnt[0];
    p.block_correct[blockIdx.x] = scor[0];
  }
}

__global__ void __launch_bounds__(kFinalizeThreads)
    flce_finalize_loss_kernel(const FinalizeParams p, int blocks) {
  __shared__ double ssum[kFinalizeThreads];
  __shared__ double sden[kFinalizeThreads];
  __shared__ long long scnt[kFinalizeThreads];
  __shared__ long long scor[kFinalizeThreads];
  double s = 0.0, dn = 0.0;
  long long c = 0, k = 0;
  for (int b = int(threadIdx.x); b < blocks; b += kFinalizeThreads) {
    s += p.block_sum[b];
    dn += p.block_wsum[b];
    c += p.block_cnt[b];
    k += p.block_correct[b];
  }
  ssum[threadIdx.x] = s;
  sden[threadIdx.x] = dn;
  scnt[threadIdx.x] = c;
  scor[threadIdx.x] = k;
  __syncthreads();
  for (int o = kFinalizeThreads / 2; o > 0; o >>= 1) {
    if (int(threadIdx.x) < o) {
      ssum[threadIdx.x] += ssum[threadIdx.x + o];
      sden[threadIdx.x] += sden[threadIdx.x + o];
      scnt[threadIdx.x] += scnt[threadIdx.x + o];
      scor[threadIdx.x] += scor[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const bool timed_out = call_timed_out(p.err);
    if (p.reduction != 2) {
      double total = ssum[0];
      if (p.reduction == 0) total = sden[0] != 0.0 ? total / sden[0] : 0.0;
      p.loss[0] = timed_out ? CUDART_NAN_F : float(total);
    }
    if (p.accuracy != nullptr)
      p.accuracy[0] = timed_out ? CUDART_NAN_F : (scnt[0] ? float(double(scor[0]) / double(scnt[0])) : 0.f);
  }
}

// One block: the mean denominator (valid rows, or the sum of their target weights; 16-byte
// vector loads of the targets) over all N rows, then g and the scalar B = g eps / V in the
// workspace header.
constexpr int kPrepThreads = 1024;

__global__ void __launch_bounds__(kPrepThreads) flce_denominator_kernel(const PrepParams p) {
  __shared__ double s_den[kPrepThreads / 32];
  const int tid = int(threadIdx.x);
  const uintptr_t addr = reinterpret_cast<uintptr_t>(p.targets);
  const flce_vec_split sp = flce_split_for_vectors(int64_t((addr & 15u) / 4u), p.N, 4);
  auto weight_of = [&](int y) -> double {
    if (y == p.ignore_index) return 0.0;
    if (p.cw == nullptr || y < 0 || y >= p.V) return 1.0;
    return double(__ldg(p.cw + y));
  };
  double den = 0.0;
  for (int64_t i = tid; i < sp.head; i += kPrepThreads) den += weight_of(p.targets[i]);
  const int4* body = reinterpret_cast<const int4*>(p.targets + sp.head);
  for (int64_t i = tid; i < sp.body / 4; i += kPrepThreads) {
    const int4 v = __ldg(body + i);
    den += weight_of(v.x) + weight_of(v.y) + weight_of(v.z) + weight_of(v.w);
  }
  for (int64_t i = sp.head + sp.body + tid; i < p.N; i += kPrepThreads) den += weight_of(p.targets[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  if ((tid & 31) == 0) s_den[tid >> 5] = den;
  __syncthreads();
  if (tid < 32) {
    double c = s_den[tid];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (tid == 0) {
      float g = *p.grad_out;
      if (p.reduction == 0) g = c != 0.0 ? float(double(g) / c) : 0.f;
      *p.gval = g;
      *p.bval = (p.gscale > 0.f ? p.gscale : g) * p.eps / float(p.V);
    }
  }
}

// Per-row coefficients for rows [0, n_rows) of `targets` / `lse` (a band of the batch):
// {A, -lse log2e, C, target column in W or kIgnoredRow} with
// A = g((1-eps) w_y + (eps/V) sum_j w_j + 2 s lse), C = g (1-eps) w_y; one 16-byte load per
// row in the gradient epilogue.
__global__ void __launch_bounds__(256) flce_coef_kernel(const PrepParams p, int n_rows) {
  const int i = int(blockIdx.x) * 256 + int(threadIdx.x);
  if (i >= n_rows) return;
  const float g = p.gscale > 0.f ? p.gscale : *p.gval;
  const float wtot = p.cw != nullptr ? *p.wtot : float(p.V);
  const int y = p.targets[i];
  float4 cf;
  if (y == p.ignore_index) {
    // A = 0 and an exponent of -inf: the epilogue's A * exp2(u log2e + y) is exactly 0 for
    // any logit u (with y = 0 a logit above ~88 would give 0 * inf = NaN)
    cf = make_float4(0.f, -CUDART_INF_F, 0.f, __int_as_float(kIgnoredRow));
  } else if (y < 0 || y >= p.V) {
    atomicOr(p.err, FLCE_DEVERR_BAD_TARGET);
    cf = make_float4(CUDART_NAN_F, 0.f, 0.f, __int_as_float(kIgnoredRow));
  } else {
    const float l = p.lse[i];
    const float wy = p.cw != nullptr ? __ldg(p.cw + y) : 1.f;
    const float a = g * ((1.f - p.eps) * wy + p.eps / float(p.V) * wtot + 2.f * p.zscale * l);
    const float c = g * (1.f - p.eps) * wy;
    // f16 band: the largest gradient entry of the row is below max(a, c) in magnitude
    if (p.gscale > 0.f && !(a <= 65504.f && c <= 65504.f)) atomicOr(p.err, FLCE_DEVERR_F16_RANGE);
    cf = make_float4(a, -l * kLog2e, c, __int_as_float(y - p.y_offset));
  }
  p.coef[i] = cf;
}

// Sum of n floats in a fixed order (one block of 1024 threads).
__global__ void __launch_bounds__(1024) flce_sum_kernel(const float* v, int n, float* out) {
  __shared__ double sh[1024];
  double s = 0.0;
  for (int i = int(threadIdx.x); i < n; i += 1024) s += double(v[i]);
  sh[threadIdx.x] = s;
  __syncthreads();
  for (int o = 512; o > 0; o >>= 1) {
    if (int(threadIdx.x) < o) sh[threadIdx.x] += sh[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = float(sh[0]);
}

// Column sums of a bf16 band: block (x, y) sums columns [256x, 256x+256) over row chunk y.
__global__ void __launch_bounds__(256) flce_colsum_partial_kernel(const ColsumParams p) {
  const int col = int(blockIdx.x) * 256 + int(threadIdx.x);
  if (col >= p.cols) return;
  const int rows_per = (p.N + p.row_chunks - 1) / p.row_chunks;
  const int r0 = int(blockIdx.y) * rows_per;
  // compacted rows: the band holds the valid rows first; the rest was not written
  const int n = p.dyn_rows != nullptr ? min(p.N, *p.dyn_rows) : p.N;
  const int r1 = min(n, r0 + rows_per);
  float s = 0.f;
  if (p.f16) {
    for (int r = r0; r < r1; ++r) s += __half2float(__ushort_as_half(p.band[size_t(r) * p.ld + col]));
  } else {
    for (int r = r0; r < r1; ++r) s += __uint_as_float(uint32_t(p.band[size_t(r) * p.ld + col]) << 16);
  }
  p.partial[size_t(blockIdx.y) * p.cols + col] = s;
}

__global__ void __launch_bounds__(256) flce_colsum_final_kernel(const ColsumParams p) {
  const int col = int(blockIdx.x) * 256 + int(threadIdx.x);
  if (col >= p.cols) return;
  float s = 0.f;
  for (int c = 0; c < p.row_chunks; ++c) s += p.partial[size_t(c) * p.cols + col];
  if (p.scale != nullptr) s *= *p.scale * p.scale_mul;
  p.out[col] = p.accumulate ? p.out[col] + s : s;
}

// Four fp32 values rounded (to nearest even) to four bf16 or f16 values.
template <bool F16>
__device__ __forceinline__ uint2 pack4_16bit(const float4 v) {
  if constexpr (F16) {
    const __half2 a = __floats2half2_rn(v.x, v.y);
    const __half2 b = __floats2half2_rn(v.z, v.w);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  } else {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  }
}

// After a timeout of a backward GEMM the casts write NaN to every dX element of the call.
template <bool F16>
__global__ void flce_cast_kernel(const float4* __restrict__ src, uint2* __restrict__ dst, size_t n4, const int* err) {
  const bool timed_out = call_timed_out(err);
  const float4 nan4 = make_float4(CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F);
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += size_t(gridDim.x) * blockDim.x)
    dst[i] = pack4_16bit<F16>(timed_out ? nan4 : src[i]);
}

// ---------------------------------------------------------------------------------
// Valid-row compaction of the backward. An ignored row's gradient is zero, so its logits
// need not be recomputed, nor its zero rows of dZ multiplied into dW and dX: the GEMMs
// run on the valid rows, gathered to the front of a scratch copy of X, and the dX
// accumulator's rows are cast back to their original places at the end.
// ---------------------------------------------------------------------------------

// The list of valid rows in order, and each row's slot in it, by several blocks: block b
// owns the rows [b R, (b + 1) R); it counts the valid rows before its range itself (a
// coalesced pass over at most N targets, cheap next to the GEMMs), then walks its range in
// tiles of 256 rows with a block-wide scan. No atomics and no waiting between blocks; the
// last block writes the count.
constexpr int kListThreads = 256;

__device__ __forceinline__ int block_sum_int(int v, int* sh) {
  const int lane = int(threadIdx.x) & 31, wid = int(threadIdx.x) >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < kListThreads / 32; ++w) t += sh[w];
  __syncthreads();
  return t;
}

__global__ void __launch_bounds__(kListThreads) flce_compact_rows_kernel(const CompactParams p, int rows_per_block) {
  __shared__ int sh[kListThreads / 32];
  __shared__ int warp_tot[kListThreads / 32];
  const int tid = int(threadIdx.x), lane = tid & 31, wid = tid >> 5;
  const int lo = min(p.N, int(blockIdx.x) * rows_per_block);
  const int hi = min(p.N, lo + rows_per_block);
  int before = 0;
  for (int i = tid; i < lo; i += kListThreads) before += p.targets[i] != p.ignore_index ? 1 : 0;
  int pos = block_sum_int(before, sh);  // slot of this block's first valid row
  for (int base = lo; base < hi; base += kListThreads) {
    const int i = base + tid;
    const int v = (i < hi && p.targets[i] != p.ignore_index) ? 1 : 0;
    int inc = v;  // inclusive scan within the warp, then over the warps' totals
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += x;
    }
    if (lane == 31) warp_tot[wid] = inc;
    __syncthreads();
    int prior = 0, tile = 0;
#pragma unroll
    for (int w = 0; w < kListThreads / 32; ++w) {
      prior += w < wid ? warp_tot[w] : 0;
      tile += warp_tot[w];
    }
    if (i < hi) {
      if (v) {
        const int at = pos + prior + inc - 1;
        p.rows[at] = i;
        p.slot[i] = at;
      } else {
        p.slot[i] = -1;
      }
    }
    pos += tile;
    __syncthreads();  // warp_tot is rewritten by the next tile
  }
  if (blockIdx.x == gridDim.x - 1 && tid == 0) *p.n_valid = pos;
}

// Row i < n_valid of the compacted operands takes X row rows[i] and its coefficients;
// rows from n_valid to the padding end (kCompactPadRows, at least one block) are zeros
// with ignored-row coefficients; rows past it are never read. One warp per row.
__global__ void __launch_bounds__(256) flce_gather_rows_kernel(const GatherParams p) {
  const int n_valid = *p.n_valid;
  int pad_end = ((n_valid > 0 ? n_valid : 1) + kCompactPadRows - 1) / kCompactPadRows * kCompactPadRows;
  if (pad_end > p.N) pad_end = p.N;
  const int lane = int(threadIdx.x) & 31;
  const int warps = int(gridDim.x) * (int(blockDim.x) >> 5);
  const int n16 = p.D / 8;  // 16-byte chunks of a row
  for (int i = int(blockIdx.x) * (int(blockDim.x) >> 5) + (int(threadIdx.x) >> 5); i < pad_end; i += warps) {
    const bool valid = i < n_valid;
    const int src = valid ? p.rows[i] : 0;
    const uint4* from = reinterpret_cast<const uint4*>(p.X) + size_t(src) * size_t(n16);
    uint4* to = reinterpret_cast<uint4*>(p.Xc) + size_t(i) * size_t(n16);
    for (int c = lane; c < n16; c += 32) to[c] = valid ? from[c] : make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0 && p.coef_c != nullptr)
      p.coef_c[i] = valid ? p.coef[src] : make_float4(0.f, -CUDART_INF_F, 0.f, __int_as_float(kIgnoredRow));
  }
}

// dX row r = the compacted accumulator's row slot[r] in 16 bits, or zeros for an ignored
// row. One warp per row.
template <bool F16>
__global__ void __launch_bounds__(256) flce_scatter_cast_kernel(const ScatterCastParams p) {
  const int lane = int(threadIdx.x) & 31;
  const int warps = int(gridDim.x) * (int(blockDim.x) >> 5);
  const int n4 = p.D / 4;
  const bool timed_out = call_timed_out(p.err);
  const float4 nan4 = make_float4(CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F);
  for (int r = int(blockIdx.x) * (int(blockDim.x) >> 5) + (int(threadIdx.x) >> 5); r < p.N; r += warps) {
    const int sl = p.slot[r];
    const float4* from = reinterpret_cast<const float4*>(p.acc) + size_t(sl < 0 ? 0 : sl) * size_t(n4);
    uint2* to = reinterpret_cast<uint2*>(p.dX) + size_t(r) * size_t(n4);
    for (int c = lane; c < n4; c += 32)
      to[c] = timed_out ? pack4_16bit<F16>(nan4) : (sl < 0 ? make_uint2(0u, 0u) : pack4_16bit<F16>(from[c]));
  }
}

// Self-test of the bounded pipeline wait: two threads wait on an mbarrier that nothing
// arrives on, with the wait the GEMMs use. One gives up after the time limit and raises
// the abort flag and FLCE_DEVERR_TIMEOUT; the other returns on the flag (or its own
// limit). Nothing else runs: no copies, no tensor memory, no cluster.
__global__ void __launch_bounds__(64) flce_wait_selftest_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const WaitCtx w{&abort_flag, err};
  if (threadIdx.x == 0 || threadIdx.x == 32) mbar_wait(&bar, 0, w);
  __syncthreads();
}

// ---------------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------------
namespace {
std::atomic<unsigned long long> g_launches{0};

// Device timing of the GEMM launches, for diagnostics: event pairs recorded around each
// launch while enabled, read (and released) by profile_read.
struct ProfRecord {
  int kind;
  cudaEvent_t start, stop;
};
std::atomic<bool> g_prof_on{false};
std::mutex g_prof_mu;
std::vector<ProfRecord> g_prof;
thread_local cudaEvent_t t_prof_start[GEMM_KINDS] = {};
}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

unsigned long long launches_so_far() { return g_launches.load(std::memory_order_relaxed); }

void profile_begin(int kind, cudaStream_t stream) {
  if (!g_prof_on.load(std::memory_order_relaxed) || kind < 0 || kind >= GEMM_KINDS) return;
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess || cudaEventRecord(e, stream) != cudaSuccess) {
    if (e) cudaEventDestroy(e);
    cudaGetLastError();
    return;
  }
  t_prof_start[kind] = e;
}

void profile_end(int kind, cudaStream_t stream) {
  if (kind < 0 || kind >= GEMM_KINDS || t_prof_start[kind] == nullptr) return;
  cudaEvent_t start = t_prof_start[kind], stop = nullptr;
  t_prof_start[kind] = nullptr;
  if (cudaEventCreate(&stop) != cudaSuccess || cudaEventRecord(stop, stream) != cudaSuccess) {
    if (stop) cudaEventDestroy(stop);
    cudaEventDestroy(start);
    cudaGetLastError();
    return;
  }
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof.push_back(ProfRecord{kind, start, stop});
}

void profile_enable(bool on) { g_prof_on.store(on, std::memory_order_relaxed); }

cudaError_t profile_read(double* ms, unsigned long long* launches) {
  std::vector<ProfRecord> recs;
  {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    recs.swap(g_prof);
  }
  for (int k = 0; k < GEMM_KINDS; ++k) {
    ms[k] = 0.0;
    launches[k] = 0;
  }
  cudaError_t first = cudaSuccess;
  for (const ProfRecord& r : recs) {
    float t = 0.f;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.start, r.stop);
    if (e == cudaSuccess) {
      ms[r.kind] += double(t);
      launches[r.kind] += 1;
    } else if (first == cudaSuccess) {
      first = e;
    }
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  return first;
}

cudaError_t launch_finalize(const FinalizeParams& p, int blocks, cudaStream_t stream) {
  flce_finalize_rows_kernel<<<blocks, kFinalizeThreads, 0, stream>>>(p);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.mode == FIN_SHARD_STATS || (p.reduction == 2 && p.accuracy == nullptr)) return e;
  flce_finalize_loss_kernel<<<1, kFinalizeThreads, 0, stream>>>(p, blocks);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_denominator(const PrepParams& p, cudaStream_t stream) {
  flce_denominator_kernel<<<1, kPrepThreads, 0, stream>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_coef(const PrepParams& p, int n_rows, cudaStream_t stream) {
  flce_coef_kernel<<<unsigned((n_rows + 255) / 256), 256, 0, stream>>>(p, n_rows);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* err, cudaStream_t stream) {
  flce_wait_selftest_kernel<<<1, 64, 0, stream>>>(err);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_sum(const float* v, int n, float* out, cudaStream_t stream) {
  flce_sum_kernel<<<1, 1024, 0, stream>>>(v, n, out);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_colsum(const ColsumParams& p, cudaStream_t stream) {
  const dim3 grid(unsigned((p.cols + 255) / 256), unsigned(p.row_chunks));
  flce_colsum_partial_kernel<<<grid, 256, 0, stream>>>(p);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  flce_colsum_final_kernel<<<unsigned((p.cols + 255) / 256), 256, 0, stream>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_compact_rows(const CompactParams& p, cudaStream_t stream) {
  // ranges of at least 1024 rows, at most 256 blocks
  int blocks = (p.N + 1023) / 1024;
  if (blocks > 256) blocks = 256;
  if (blocks < 1) blocks = 1;
  const int per = (p.N + blocks - 1) / blocks;
  flce_compact_rows_kernel<<<blocks, kListThreads, 0, stream>>>(p, per);
  count_launch();
  return cudaGetLastError();
}

namespace {
// warp-per-row kernels: 8 warps a block, up to 8 blocks an SM, no more blocks than rows need
unsigned row_blocks(int rows, int num_sms) {
  const int need = (rows + 7) / 8, cap = num_sms * 8;
  return unsigned(need < 1 ? 1 : (need < cap ? need : cap));
}
}  // namespace

cudaError_t launch_gather_rows(const GatherParams& p, int num_sms, cudaStream_t stream) {
  flce_gather_rows_kernel<<<row_blocks(p.N, num_sms), 256, 0, stream>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_scatter_cast(const ScatterCastParams& p, int num_sms, cudaStream_t stream) {
  if (p.f16)
    flce_scatter_cast_kernel<true><<<row_blocks(p.N, num_sms), 256, 0, stream>>>(p);
  else
    flce_scatter_cast_kernel<false><<<row_blocks(p.N, num_sms), 256, 0, stream>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_cast_16bit(const float* src, void* dst, size_t n, bool f16, int num_sms, const int* err,
                              cudaStream_t stream) {
  const size_t n4 = n / 4;
  size_t blocks = (n4 + 255) / 256;
  const size_t cap = size_t(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  if (f16)
    flce_cast_kernel<true><<<unsigned(blocks), 256, 0, stream>>>(reinterpret_cast<const float4*>(src),
                                                                 reinterpret_cast<uint2*>(dst), n4, err);
  else
    flce_cast_kernel<false><<<unsigned(blocks), 256, 0, stream>>>(reinterpret_cast<const float4*>(src),
                                                                  reinterpret_cast<uint2*>(dst), n4, err);
  count_launch();
  return cudaGetLastError();
}

}  // namespace flce
