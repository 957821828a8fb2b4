// flce_small.cu -- the bandwidth/latency-bound helper kernels of fused linear
// cross-entropy: the forward finalize (combine the vocabulary splits into lse, form the
// row losses, reduce them in a fixed order), the backward prep (valid-row count and
// per-row gradient coefficients) and the fp32 -> bf16 cast of dX.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "flce_internal.h"
#include "vec_split.h"

namespace flce {

namespace {
constexpr float kLog2e = 1.4426950408889634f;
}

// ---------------------------------------------------------------------------------
// ---------------------------------------------------------------------------------

// Combine the S partial statistics of each row into lse, form the row loss and
// reduce it deterministically (per-block fp64 partial sums, then one block).
__global__ void __launch_bounds__(kFinalizeThreads)
    flce_finalize_rows_kernel(const FinalizeParams p) {
  const int row = int(blockIdx.x) * kFinalizeThreads + int(threadIdx.x);
  double contrib = 0.0;
  int valid = 0;
  if (row < p.N) {
    float M = -CUDART_INF_F;
    for (int s = 0; s < p.S; ++s) M = fmaxf(M, p.part_m[size_t(s) * p.N + row]);
    float d = 0.f, sz = 0.f;
    for (int s = 0; s < p.S; ++s) {
      const size_t o = size_t(s) * p.N + row;
      d += p.part_d[o] * exp2f((p.part_m[o] - M) * kLog2e);
      sz += p.part_s[o];
    }
    const float lse = M + logf(d);
    p.lse[row] = lse;
    const int y = p.targets[row];
    float ell = 0.f;
    if (y != p.ignore_index) {
      valid = 1;
      if (y < 0 || y >= p.V) {
        atomicOr(p.err, FLCE_DEVERR_BAD_TARGET);
        ell = CUDART_NAN_F;
      } else {
        const float zy = p.tgt[row];
        ell = (1.f - p.eps) * (lse - zy) + p.zscale * lse * lse;
        if (p.eps != 0.f) ell += p.eps * (lse - sz / float(p.V));
      }
    }
    if (p.reduction == 2) p.loss[row] = ell;
    contrib = double(ell);
  }
  if (p.reduction == 2) return;
  // fixed-order block reduction
  __shared__ double ssum[kFinalizeThreads];
  __shared__ int scnt[kFinalizeThreads];
  ssum[threadIdx.x] = contrib;
  scnt[threadIdx.x] = valid;
  __syncthreads();
  for (int o = kFinalizeThreads / 2; o > 0; o >>= 1) {
    if (int(threadIdx.x) < o) {
      ssum[threadIdx.x] += ssum[threadIdx.x + o];
      scnt[threadIdx.x] += scnt[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.block_sum[blockIdx.x] = ssum[0];
    p.block_cnt[blockIdx.x] = scnt[0];
  }
}

__global__ void __launch_bounds__(kFinalizeThreads)
    flce_finalize_loss_kernel(const FinalizeParams p, int blocks) {
  __shared__ double ssum[kFinalizeThreads];
  __shared__ long long scnt[kFinalizeThreads];
  double s = 0.0;
  long long c = 0;
  for (int b = int(threadIdx.x); b < blocks; b += kFinalizeThreads) {
    s += p.block_sum[b];
    c += p.block_cnt[b];
  }
  ssum[threadIdx.x] = s;
  scnt[threadIdx.x] = c;
  __syncthreads();
  for (int o = kFinalizeThreads / 2; o > 0; o >>= 1) {
    if (int(threadIdx.x) < o) {
      ssum[threadIdx.x] += ssum[threadIdx.x + o];
      scnt[threadIdx.x] += scnt[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    double total = ssum[0];
    if (p.reduction == 0) total = scnt[0] ? total / double(scnt[0]) : 0.0;
    p.loss[0] = float(total);
  }
}

// One block: count valid rows (16-byte vector loads of the targets), form g, then the
// per-row coefficients {a = g(1 + 2 s lse), -lse log2e, b = g eps / V, target} the
// gradient epilogue reads with one 16-byte load per row.
constexpr int kPrepThreads = 1024;

__global__ void __launch_bounds__(kPrepThreads) flce_prep_kernel(const PrepParams p) {
  __shared__ int s_cnt[kPrepThreads / 32];
  __shared__ float s_g;
  const int tid = int(threadIdx.x);
  const uintptr_t addr = reinterpret_cast<uintptr_t>(p.targets);
  const flce_vec_split sp = flce_split_for_vectors(int64_t((addr & 15u) / 4u), p.N, 4);
  int cnt = 0;
  for (int64_t i = tid; i < sp.head; i += kPrepThreads) cnt += (p.targets[i] != p.ignore_index);
  const int4* body = reinterpret_cast<const int4*>(p.targets + sp.head);
  for (int64_t i = tid; i < sp.body / 4; i += kPrepThreads) {
    const int4 v = __ldg(body + i);
    cnt += (v.x != p.ignore_index) + (v.y != p.ignore_index) + (v.z != p.ignore_index) + (v.w != p.ignore_index);
  }
  for (int64_t i = sp.head + sp.body + tid; i < p.N; i += kPrepThreads) cnt += (p.targets[i] != p.ignore_index);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((tid & 31) == 0) s_cnt[tid >> 5] = cnt;
  __syncthreads();
  if (tid < 32) {
    int c = s_cnt[tid];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (tid == 0) {
      float g = *p.grad_out;
      if (p.reduction == 0) g = c ? g / float(c) : 0.f;
      s_g = g;
      *p.cval = g * (1.f - p.eps);
    }
  }
  __syncthreads();
  const float g = s_g;
  const float b = g * p.eps / float(p.V);
  for (int i = tid; i < p.N; i += kPrepThreads) {
    const int y = p.targets[i];
    float4 cf;
    if (y == p.ignore_index) {
      cf = make_float4(0.f, 0.f, 0.f, __int_as_float(-1));
    } else if (y < 0 || y >= p.V) {
      atomicOr(p.err, FLCE_DEVERR_BAD_TARGET);
      cf = make_float4(CUDART_NAN_F, 0.f, 0.f, __int_as_float(-1));
    } else {
      const float l = p.lse[i];
      cf = make_float4(g * (1.f + 2.f * p.zscale * l), -l * kLog2e, b, __int_as_float(y));
    }
    p.coef[i] = cf;
  }
}

__global__ void flce_cast_bf16_kernel(const float4* __restrict__ src, uint2* __restrict__ dst, size_t n4) {
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += size_t(gridDim.x) * blockDim.x) {
    const float4 v = src[i];
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    dst[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  }
}

// ---------------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------------
cudaError_t launch_finalize(const FinalizeParams& p, int blocks, cudaStream_t stream) {
  flce_finalize_rows_kernel<<<blocks, kFinalizeThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.reduction == 2) return e;
  flce_finalize_loss_kernel<<<1, kFinalizeThreads, 0, stream>>>(p, blocks);
  return cudaGetLastError();
}

cudaError_t launch_prep(const PrepParams& p, cudaStream_t stream) {
  flce_prep_kernel<<<1, kPrepThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_cast_bf16(const float* src, void* dst, size_t n, int num_sms, cudaStream_t stream) {
  const size_t n4 = n / 4;
  size_t blocks = (n4 + 255) / 256;
  const size_t cap = size_t(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  flce_cast_bf16_kernel<<<unsigned(blocks), 256, 0, stream>>>(reinterpret_cast<const float4*>(src),
                                                              reinterpret_cast<uint2*>(dst), n4);
  return cudaGetLastError();
}

}  // namespace flce
