// flce_gemm.cu -- the tensor-core kernels of fused linear cross-entropy on sm_103a.
//
// All four GEMMs share one warp-specialised, persistent skeleton:
//   warp 0      : TMA producer. One elected lane streams A and B K-blocks (64 bf16
//                 deep, 128-byte swizzled) into a 4-stage shared-memory ring.
//   warp 1      : MMA issuer. Allocates 512 TMEM columns (two 128x256 fp32
//                 accumulators), issues tcgen05.mma (M=128, N=256, K=16) per stage
//                 and commits each stage back to the producer and each finished
//                 accumulator to the epilogue.
//   warps 2..5  : epilogue. 128 threads, thread r owns TMEM lane r = output row r,
//                 so every per-row reduction is thread-local. While they drain one
//                 accumulator the MMA warp fills the other.
//
// The epilogues:
//   forward   : online softmax over the tile's vocabulary columns (running max m,
//               sum of exp(z - m), sum of z) and capture of the target logit; the
//               logits never leave the chip. ("Cutting LLM Memory by 84%: A Deep
//               Dive into Fused Kernels", "Definition and Forward Pass" and
//               "Kernel Implementation"; Liger-Kernel PR #1291 "Summary": a
//               store-free forward that keeps only the per-row LSE and target logit.)
//   gradient  : recomputed logits -> G = g[p(1+2s lse) - (1-eps) onehot - eps/V] in
//               registers, rounded to bf16 and stored by TMA into the gradient band.
//               ("Cross-Entropy" and "Fused Linear Cross-Entropy" of the same post;
//               the smoothing rule of TransformerEngine PR #995's backward kernel.)
//   dW / dX   : fp32 accumulator -> shared memory -> TMA store (dW, each block written
//               once) or TMA element-wise add (dX accumulation across vocabulary
//               bands, no atomics on the same element within a launch).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "flce_internal.h"
#include "sm103_ptx.cuh"
#include "vec_split.h"

namespace flce {

constexpr float kLog2e = 1.4426950408889634f;

enum : int { TILE_FIRST = 1, TILE_LAST = 2 };

struct Tile {
  int a_row;   // A operand: first M row (K-major) or first M column (MN-major)
  int b_row;   // B operand: first N row (K-major) or first N column (MN-major)
  int a_k0;    // K coordinate of the first K block in A
  int b_k0;    // ... and in B
  int num_kb;  // number of 64-wide K blocks
  int aux;     // forward: vocabulary range index of the partial statistics
  int flags;
};

// ---------------------------------------------------------------------------------
// Tile schedules (every role of a CTA walks the same sequence)
// ---------------------------------------------------------------------------------

// Forward: the grid is gN row tiles x S vocabulary ranges. CTA c keeps row-tile
// offset c % gN and walks groups of gN row tiles; in group g it covers vocabulary
// range (c / gN + g) mod S, so the extra tile of the longer ranges rotates among
// CTAs. Running statistics stay in registers across a range and are written once per
// (row, range).
struct FwdSched {
  int n_tiles, v_tiles, gN, S, num_kb;
  int n_off, split;
  int g, vt, vt_end, range, n_tile;
  bool first;

  __device__ explicit FwdSched(const FwdParams& p)
      : n_tiles(p.n_tiles), v_tiles(p.v_tiles), gN(p.gN), S(p.S), num_kb(p.num_kb),
        n_off(int(blockIdx.x) % p.gN), split(int(blockIdx.x) / p.gN), g(-1), vt(0), vt_end(0), range(0),
        n_tile(0), first(false) {}

  __device__ bool next(Tile& t) {
    if (vt >= vt_end) {
      ++g;
      n_tile = g * gN + n_off;
      if (n_tile >= n_tiles) return false;
      range = (split + g) % S;
      vt = int((long long)range * v_tiles / S);
      vt_end = int((long long)(range + 1) * v_tiles / S);
      if (vt >= vt_end) return false;  // S <= v_tiles on the host, so never taken
      first = true;
    }
    t.a_row = n_tile * kBM;
    t.b_row = vt * kBN;
    t.a_k0 = 0;
    t.b_k0 = 0;
    t.num_kb = num_kb;
    t.aux = range;
    t.flags = (first ? TILE_FIRST : 0) | (vt + 1 == vt_end ? TILE_LAST : 0);
    first = false;
    ++vt;
    return true;
  }
};

// Static round-robin walk for the backward GEMMs. Tile index i = major * minor_count + minor.
//   WALK_GRAD: major = row tile of X (128 rows), minor = 256-column vocabulary tile of the band.
//   WALK_DW  : major = 256-column vocabulary tile, minor = 128-row tile of D.
//   WALK_DX  : major = row tile of the band (128 rows), minor = 256-column tile of D.
template <int KIND>
struct WalkSched {
  WalkParams w;
  int i;
  __device__ explicit WalkSched(const WalkParams& p) : w(p), i(int(blockIdx.x)) {}
  __device__ bool next(Tile& t) {
    if (i >= w.total_tiles) return false;
    const int major = i / w.tiles_minor;
    const int minor = i - major * w.tiles_minor;
    if (KIND == WALK_GRAD) {
      t.a_row = major * kBM;
      t.b_row = w.b_row_off + minor * kBN;
    } else if (KIND == WALK_DW) {
      t.a_row = minor * kBM;
      t.b_row = w.b_row_off + major * kBN;
    } else {
      t.a_row = major * kBM;
      t.b_row = w.b_row_off + minor * kBN;
    }
    t.a_k0 = w.a_k0;
    t.b_k0 = w.b_k0;
    t.num_kb = w.num_kb;
    t.aux = 0;
    t.flags = TILE_FIRST | TILE_LAST;
    i += int(gridDim.x);
    return true;
  }
};

// ---------------------------------------------------------------------------------
// Shared memory and the two async roles
// ---------------------------------------------------------------------------------
struct Smem {
  uint8_t* stage;      // kStages x (A 16 KB | B 32 KB), 1024-byte aligned
  uint8_t* staging;    // epilogue store boxes, 16 KB each
  uint64_t* full;      // [kStages] TMA -> MMA
  uint64_t* empty;     // [kStages] MMA -> TMA
  uint64_t* tfull;     // [2] accumulator ready for the epilogue
  uint64_t* tempty;    // [2] accumulator drained
  uint64_t* drain;     // MMA completion on abort
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  volatile int* epi_go;  // [2]
};

__device__ __forceinline__ Smem carve_smem(uint8_t* raw, int staging_bufs) {
  Smem s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.stage = base;
  s.staging = base + kStages * kStageBytes;
  uint8_t* b = s.staging + staging_bufs * kStagingBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(b);
  s.full = bars;
  s.empty = bars + kStages;
  s.tfull = bars + 2 * kStages;
  s.tempty = bars + 2 * kStages + 2;
  s.drain = bars + 2 * kStages + 4;
  uint32_t* words = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
  s.tmem_slot = words;
  s.abort_flag = reinterpret_cast<volatile int*>(words + 1);
  s.epi_go = reinterpret_cast<volatile int*>(words + 2);
  return s;
}

template <bool A_MN, bool B_MN>
__device__ __forceinline__ void load_stage(uint8_t* sa, uint8_t* sb, const CUtensorMap* tma, const CUtensorMap* tmb,
                                           uint64_t* bar, const Tile& t, int kb) {
  const int ka = t.a_k0 + kb * kBK;
  const int kbb = t.b_k0 + kb * kBK;
  if (!A_MN) {
    tma_load_2d(sa, tma, bar, ka, t.a_row);  // box {64 K, 128 rows}
  } else {
#pragma unroll
    for (int j = 0; j < kBM / 64; ++j) tma_load_2d(sa + j * 8192, tma, bar, t.a_row + 64 * j, ka);  // {64 M, 64 K}
  }
  if (!B_MN) {
    tma_load_2d(sb, tmb, bar, kbb, t.b_row);  // box {64 K, 256 rows}
  } else {
#pragma unroll
    for (int j = 0; j < kBN / 64; ++j) tma_load_2d(sb + j * 8192, tmb, bar, t.b_row + 64 * j, kbb);  // {64 N, 64 K}
  }
}

template <bool A_MN, bool B_MN>
__device__ __forceinline__ void mma_stage(uint32_t d_tmem, uint32_t sa, uint32_t sb, bool acc_first) {
  constexpr uint32_t idesc = make_idesc_bf16(kBM, kBN, A_MN, B_MN);
#pragma unroll
  for (int kk = 0; kk < kBK / 16; ++kk) {
    // K-major: advance 16 elements = 32 bytes inside the swizzled 128-byte row.
    // MN-major: advance 16 K-rows = 2048 bytes; MN chunks of 64 elements are 8 KB apart.
    const uint64_t ad = A_MN ? make_sdesc_sw128(sa + kk * 2048, 8192, 1024) : make_sdesc_sw128(sa + kk * 32, 16, 1024);
    const uint64_t bd = B_MN ? make_sdesc_sw128(sb + kk * 2048, 8192, 1024) : make_sdesc_sw128(sb + kk * 32, 16, 1024);
    tc_mma_bf16(d_tmem, ad, bd, idesc, (acc_first || kk > 0) ? 1u : 0u);
  }
}

template <bool A_MN, bool B_MN, class Sched, class SP>
__device__ __forceinline__ void producer_role(const Smem& s, const CUtensorMap* tma, const CUtensorMap* tmb,
                                              const SP& sp, const WaitCtx& w) {
  Sched sched(sp);
  Tile t;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0, last_parity = 0;
  bool ok = true;
  while (ok && sched.next(t)) {
    for (int kb = 0; kb < t.num_kb; ++kb) {
      if (!mbar_wait(&s.empty[stage], phase ^ 1u, w)) { ok = false; break; }
      mbar_arrive_expect_tx(&s.full[stage], kStageBytes);
      uint8_t* sa = s.stage + stage * kStageBytes;
      load_stage<A_MN, B_MN>(sa, sa + kABytes, tma, tmb, &s.full[stage], t, kb);
      issued |= 1u << stage;
      last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == kStages) { stage = 0; phase ^= 1u; }
    }
  }
  if (!ok) {
    // Aborting: let every copy this thread started land before the CTA exits.
    for (int st = 0; st < kStages; ++st)
      if (issued & (1u << st)) mbar_wait_drain(&s.full[st], (last_parity >> st) & 1u);
  }
}

template <bool A_MN, bool B_MN, class Sched, class SP>
__device__ __forceinline__ void mma_role(const Smem& s, uint32_t tmem_base, const SP& sp, const WaitCtx& w) {
  Sched sched(sp);
  Tile t;
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool ok = true;
  bool issued_any = false;
  while (ok && sched.next(t)) {
    if (!mbar_wait(&s.tempty[acc], acc_phase ^ 1u, w)) { ok = false; break; }
    tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + uint32_t(acc * kBN);
    for (int kb = 0; kb < t.num_kb; ++kb) {
      if (!mbar_wait(&s.full[stage], phase, w)) { ok = false; break; }
      tc_fence_after_sync();
      const uint32_t sa = smem_addr(s.stage + stage * kStageBytes);
      mma_stage<A_MN, B_MN>(d_tmem, sa, sa + kABytes, kb > 0);
      issued_any = true;
      tc_commit(&s.empty[stage]);
      if (++stage == kStages) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    tc_commit(&s.tfull[acc]);
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
  if (!ok && issued_any) {
    // Aborting: wait for the MMAs already issued before TMEM is released.
    tc_commit(s.drain);
    mbar_wait_drain(s.drain, 0);
  }
}

// Epilogue thread bookkeeping: thread 0 of the epilogue waits on the accumulator
// barrier (bounded) and tells the other 127 through shared memory, so that every
// epilogue thread takes the same path and the named barriers below cannot deadlock.
__device__ __forceinline__ bool epi_acquire(const Smem& s, int acc, uint32_t acc_phase, int epi_tid,
                                            const WaitCtx& w) {
  if (epi_tid == 0) {
    const bool ok = mbar_wait(&s.tfull[acc], acc_phase, w) && !*s.abort_flag;
    s.epi_go[acc] = ok ? 1 : 0;
  }
  named_barrier_sync(1, kEpiThreads);
  const bool go = s.epi_go[acc] != 0;
  if (go) tc_fence_after_sync();
  return go;
}

__device__ __forceinline__ void epi_release(const Smem& s, int acc) {
  tc_fence_before_sync();
  mbar_arrive(&s.tempty[acc]);
}

// ---------------------------------------------------------------------------------
// Forward GEMM: logits tile -> online softmax statistics (never stored)
// ---------------------------------------------------------------------------------
struct RowStats {
  float m, d, sz, zy;
  bool cap;
};

template <bool kMasked>
__device__ __forceinline__ void online_update(RowStats& st, const uint32_t (&r)[32], int col0, int V, int y,
                                              bool want_sum) {
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    v[j] = __uint_as_float(r[j]);
    if (kMasked && col0 + j >= V) v[j] = -CUDART_INF_F;
  }
  // target logit: only the tile that holds column y writes it
  const int rel = y - col0;
  if (static_cast<unsigned>(rel) < 32u) {
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) z = (j == rel) ? v[j] : z;
    st.zy = z;
    st.cap = true;
  }
  float cm = v[0];
#pragma unroll
  for (int j = 1; j < 32; ++j) cm = fmaxf(cm, v[j]);
  const float nm = fmaxf(st.m, cm);
  const float scale = exp2f((st.m - nm) * kLog2e);
  const float nml = nm * kLog2e;
  float e0 = 0.f, e1 = 0.f;
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    e0 += exp2f(fmaf(v[j], kLog2e, -nml));
    e1 += exp2f(fmaf(v[j + 1], kLog2e, -nml));
  }
  st.d = st.d * scale + (e0 + e1);
  st.m = nm;
  if (want_sum) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      if (!kMasked) {
        s0 += v[j];
        s1 += v[j + 1];
      } else {
        s0 += (col0 + j < V) ? v[j] : 0.f;
        s1 += (col0 + j + 1 < V) ? v[j + 1] : 0.f;
      }
    }
    st.sz += s0 + s1;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    flce_forward_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem s = carve_smem(smem_raw, 0);
  const int warp = int(threadIdx.x) >> 5;
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], kEpiThreads);
    }
    mbar_init(s.drain, 1);
    *s.abort_flag = 0;
    s.epi_go[0] = 0;
    s.epi_go[1] = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(s.tmem_slot, 512);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *s.tmem_slot;
  const WaitCtx w{s.abort_flag, p.err};

  if (warp == 0) {
    if (lane == 0) producer_role<false, true, FwdSched>(s, &tmA, &tmB, p, w);
  } else if (warp == 1) {
    if (lane == 0) mma_role<false, true, FwdSched>(s, tmem_base, p, w);
  } else {
    const int epi_tid = int(threadIdx.x) - 64;
    const int r = 32 * (warp & 3) + int(lane);  // TMEM lane = tile row
    const uint32_t lane_addr = tmem_base + (uint32_t(32 * (warp & 3)) << 16);
    FwdSched sched(p);
    Tile t;
    int acc = 0;
    uint32_t acc_phase = 0;
    RowStats st{-CUDART_INF_F, 0.f, 0.f, 0.f, false};
    int row = 0, y = -1;
    const bool want_sum = p.want_sum_z != 0;
    while (sched.next(t)) {
      if (!epi_acquire(s, acc, acc_phase, epi_tid, w)) break;
      if (t.flags & TILE_FIRST) {
        row = t.a_row + r;
        y = (row < p.N) ? __ldg(p.targets + row) : -1;
        st = RowStats{-CUDART_INF_F, 0.f, 0.f, 0.f, false};
      }
      const uint32_t taddr = lane_addr + uint32_t(acc * kBN);
      const bool tail_tile = t.b_row + kBN > p.V;
#pragma unroll 1
      for (int c = 0; c < kBN; c += 64) {
        uint32_t r0[32], r1[32];
        tmem_ld_32cols(taddr + uint32_t(c), r0);
        tmem_ld_32cols(taddr + uint32_t(c + 32), r1);
        tc_wait_ld();
        if (c + 64 == kBN) epi_release(s, acc);
        const int col0 = t.b_row + c;
        if (!tail_tile) {
          online_update<false>(st, r0, col0, p.V, y, want_sum);
          online_update<false>(st, r1, col0 + 32, p.V, y, want_sum);
        } else {
          if (col0 < p.V) online_update<true>(st, r0, col0, p.V, y, want_sum);
          if (col0 + 32 < p.V) online_update<true>(st, r1, col0 + 32, p.V, y, want_sum);
        }
      }
      if ((t.flags & TILE_LAST) && row < p.N) {
        const size_t o = size_t(t.aux) * size_t(p.N) + size_t(row);
        p.part_m[o] = st.m;
        p.part_d[o] = st.d;
        p.part_s[o] = st.sz;
        if (st.cap) p.tgt[row] = st.zy;
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

// ---------------------------------------------------------------------------------
// Backward GEMMs (gradient band, dW, dX)
// ---------------------------------------------------------------------------------

// Write 16 bytes per chunk q (0..7) of row r of a 128-byte-swizzled 128 x 128 B box.
__device__ __forceinline__ void staging_write_row(uint8_t* box, int r, const uint4 (&chunks)[8]) {
  uint8_t* row = box + r * 128;
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<uint4*>(row + ((q ^ (r & 7)) << 4)) = chunks[q];
}

// Stage one box and hand it to TMA. `box_idx` counts boxes across the CTA's lifetime;
// buffers alternate so that the copy of box i-1 overlaps the writes of box i.
template <class WriteFn>
__device__ __forceinline__ void epi_store_box(const Smem& s, int epi_tid, uint32_t box_idx, WriteFn&& write,
                                              const CUtensorMap* tm, int x, int y, bool reduce_add) {
  uint8_t* box = s.staging + (box_idx & 1u) * kStagingBytes;
  if (epi_tid == 0) bulk_wait_group_read<1>();  // the copy that last read this buffer is done
  named_barrier_sync(1, kEpiThreads);
  write(box);
  fence_proxy_async_smem();
  named_barrier_sync(1, kEpiThreads);
  if (epi_tid == 0) {
    if (reduce_add)
      tma_reduce_add_2d(tm, box, x, y);
    else
      tma_store_2d(tm, box, x, y);
    bulk_commit_group();
  }
}

template <bool A_MN, bool B_MN, int KIND, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    flce_walk_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmC, const WalkParams wp, const GradEpiParams gp,
                          const StoreEpiParams sp) {
  extern __shared__ uint8_t smem_raw[];
  const Smem s = carve_smem(smem_raw, 2);
  const int warp = int(threadIdx.x) >> 5;
  const uint32_t lane = lane_id();
  int* err = (EPI == 0) ? gp.err : sp.err;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], kEpiThreads);
    }
    mbar_init(s.drain, 1);
    *s.abort_flag = 0;
    s.epi_go[0] = 0;
    s.epi_go[1] = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(s.tmem_slot, 512);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *s.tmem_slot;
  const WaitCtx w{s.abort_flag, err};

  if (warp == 0) {
    if (lane == 0) producer_role<A_MN, B_MN, WalkSched<KIND>>(s, &tmA, &tmB, wp, w);
  } else if (warp == 1) {
    if (lane == 0) mma_role<A_MN, B_MN, WalkSched<KIND>>(s, tmem_base, wp, w);
  } else {
    const int epi_tid = int(threadIdx.x) - 64;
    const int r = 32 * (warp & 3) + int(lane);
    const uint32_t lane_addr = tmem_base + (uint32_t(32 * (warp & 3)) << 16);
    WalkSched<KIND> sched(wp);
    Tile t;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t box_idx = 0;
    while (sched.next(t)) {
      if (!epi_acquire(s, acc, acc_phase, epi_tid, w)) break;
      const uint32_t taddr = lane_addr + uint32_t(acc * kBN);
      if (EPI == 0) {
        // G = a * exp2(z*log2e - lse*log2e) - b - [col == y] c, zero outside the vocabulary.
        const int row = t.a_row + r;
        float4 cf = make_float4(0.f, 0.f, 0.f, __int_as_float(-1));
        if (row < gp.N) cf = __ldg(gp.coef + row);
        const float cval = __ldg(gp.cval);
        const int y = __float_as_int(cf.w);
#pragma unroll 1
        for (int c = 0; c < kBN; c += 64) {
          uint32_t r0[32], r1[32];
          tmem_ld_32cols(taddr + uint32_t(c), r0);
          tmem_ld_32cols(taddr + uint32_t(c + 32), r1);
          tc_wait_ld();
          if (c + 64 == kBN) epi_release(s, acc);
          const int col0 = t.b_row + c;  // global vocabulary column
          uint4 chunks[8];
          uint32_t* packed = reinterpret_cast<uint32_t*>(chunks);
#pragma unroll
          for (int j = 0; j < 64; j += 2) {
            const float z0 = __uint_as_float(j < 32 ? r0[j] : r1[j - 32]);
            const float z1 = __uint_as_float(j + 1 < 32 ? r0[j + 1] : r1[j + 1 - 32]);
            float g0 = cf.x * exp2f(fmaf(z0, kLog2e, cf.y)) - cf.z;
            float g1 = cf.x * exp2f(fmaf(z1, kLog2e, cf.y)) - cf.z;
            if (col0 + j == y) g0 -= cval;
            if (col0 + j + 1 == y) g1 -= cval;
            if (col0 + j >= gp.V) g0 = 0.f;
            if (col0 + j + 1 >= gp.V) g1 = 0.f;
            const __nv_bfloat162 h = __floats2bfloat162_rn(g0, g1);
            packed[j >> 1] = *reinterpret_cast<const uint32_t*>(&h);
          }
          epi_store_box(
              s, epi_tid, box_idx++, [&](uint8_t* box) { staging_write_row(box, r, chunks); }, &tmC,
              col0 - gp.chunk_v0, t.a_row, false);
        }
      } else {
        // fp32 accumulator -> dW (store) or dX accumulator (store / add), 32 columns per box.
#pragma unroll 1
        for (int c = 0; c < kBN; c += 32) {
          uint32_t r0[32];
          tmem_ld_32cols(taddr + uint32_t(c), r0);
          tc_wait_ld();
          if (c + 32 == kBN) epi_release(s, acc);
          uint4 chunks[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) chunks[q] = make_uint4(r0[4 * q], r0[4 * q + 1], r0[4 * q + 2], r0[4 * q + 3]);
          epi_store_box(
              s, epi_tid, box_idx++, [&](uint8_t* box) { staging_write_row(box, r, chunks); }, &tmC,
              sp.x_off + t.b_row + c, t.a_row, sp.reduce_add != 0);
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (epi_tid == 0) bulk_wait_group<0>();  // every store has landed before the CTA exits
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

// ---------------------------------------------------------------------------------
// Small kernels: forward finalize, backward row coefficients, dX cast
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
template <class K>
static cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
}

cudaError_t launch_forward_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const FwdParams& p,
                                cudaStream_t stream) {
  const size_t smem = gemm_smem_bytes(0);
  cudaError_t e = set_smem(flce_forward_gemm_kernel, smem);
  if (e != cudaSuccess) return e;
  flce_forward_gemm_kernel<<<p.gN * p.S, kThreads, smem, stream>>>(tmA, tmB, p);
  return cudaGetLastError();
}

template <bool A_MN, bool B_MN, int KIND, int EPI>
static cudaError_t launch_walk(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                               const WalkParams& w, const GradEpiParams& g, const StoreEpiParams& s, int grid,
                               cudaStream_t stream) {
  auto kern = flce_walk_gemm_kernel<A_MN, B_MN, KIND, EPI>;
  const size_t smem = gemm_smem_bytes(2);
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(tmA, tmB, tmC, w, g, s);
  return cudaGetLastError();
}

cudaError_t launch_grad_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                             const WalkParams& w, const GradEpiParams& e, int grid, cudaStream_t stream) {
  StoreEpiParams unused{0, 0, e.err};
  return launch_walk<false, true, WALK_GRAD, 0>(tmA, tmB, tmC, w, e, unused, grid, stream);
}

cudaError_t launch_dw_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const WalkParams& w, const StoreEpiParams& e, int grid, cudaStream_t stream) {
  GradEpiParams unused{nullptr, nullptr, 0, 0, 0, e.err};
  return launch_walk<true, true, WALK_DW, 1>(tmA, tmB, tmC, w, unused, e, grid, stream);
}

cudaError_t launch_dx_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const WalkParams& w, const StoreEpiParams& e, int grid, cudaStream_t stream) {
  GradEpiParams unused{nullptr, nullptr, 0, 0, 0, e.err};
  return launch_walk<false, false, WALK_DX, 1>(tmA, tmB, tmC, w, unused, e, grid, stream);
}

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
