/*
 * fa_bwd.cuh -- attention backward pass on sm_103a (fp16 / bf16, D = 64 or 128).
 *
 * Given Q, K, V, the forward output O, the upstream gradient dO and the
 * per-row log-sum-exp of the forward, it computes
 *
 *     P  = exp(scale * Q K^T - lse)        (recomputed tile by tile)
 *     dV = P^T dO,   dP = dO V^T,   dS = P * (dP - rowsum(dO * O))
 *     dQ = scale * dS K,   dK = scale * dS^T Q
 *
 * -- the chain rule through the reference attention of "ops-transformer
 * FlashAttention build and tuning" (section 4.3), with the backward dQ loop
 * over key/value blocks that the Hygon retrospective describes (defect 13).
 * rowsum(dO * O) equals rowsum(P * dP) when O = P V; it is computed once per
 * row by a small kernel and stored, with lse * log2(e), in a workspace.
 *
 * Two persistent warp-specialised kernels, each with its accumulators in
 * tensor memory (TMEM) and every product on the tcgen05 tensor cores:
 *
 *   fa_bwd_dq_kernel   -- one 128-row query tile per work unit, K/V blocks
 *                          streamed: S = Q K^T, dP = dO V^T (both SS), then
 *                          dQ += dS K (A = dS from TMEM, B = K MN-major).
 *   fa_bwd_dkdv_kernel -- one 128-row key/value tile per work unit, the query
 *                          tiles of every query head that reads it streamed:
 *                          S^T = K Q^T, dP^T = V dO^T (SS), then dV += P^T dO
 *                          and dK += dS^T Q (A from TMEM, B MN-major).
 *
 * Splitting dQ from dK/dV costs two recomputed products per tile pair but
 * needs no atomics and keeps every result deterministic; with D = 128 the
 * dK/dV kernel already fills all 512 TMEM columns (S^T, dP^T, dV, dK).
 *
 * Warp roles (512 threads): warps 0-7 compute P / dS (warp w serves TMEM lane
 * quarter w % 4 and column half w / 4), warp 8 is the TMA producer, warp 9
 * issues the MMAs (each role run by its whole warp, one elected lane issuing)
 * and warps 12-15 run the epilogue: they read a unit's accumulators out of
 * TMEM, hand them back, and write them out while the next unit's products
 * run.  Consecutive units overlap further: Q / dO (dQ kernel) and K / V (dK/dV
 * kernel) are reloaded as soon as the previous unit's last products that read
 * them are done.  Every wait is bounded (see fa_ptx.cuh).
 */
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <cstdint>

#include "fa_ptx.cuh"
#include "fa_tmem_io.cuh"

namespace fa {
namespace bwd {

constexpr int kF16 = 0, kBF16 = 1;  // element type codes (as the forward's)
// Warp roles (512 threads, four warpgroups): warps 0-7 compute P and dS,
// warp 8 is the TMA producer, warp 9 issues the MMAs (10 and 11 idle), warps
// 12-15 run the epilogue -- read the accumulators out of TMEM, hand them back
// and write them out while the next unit's products run.
constexpr int kThreads = 512;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kEpiWarp0 = 12;
// Registers per thread by warpgroup (setmaxnreg): launched with 128 each.
constexpr uint32_t kRegSoftmax = 168, kRegControl = 72, kRegEpilogue = 104;
static_assert(2 * kRegSoftmax + kRegControl + kRegEpilogue == 4 * 128, "register budget");
constexpr uint32_t kTmemCols = 512;

struct BwdParams {
  int64_t B, H, H_kv, S_q, S_kv;
  int64_t S_q_pad;        // rows per head of the lse2 / dsum arrays (n_q_tiles * 128)
  int32_t kv_group;       // query heads per key/value head
  int32_t n_q_tiles, n_kv_tiles;
  int32_t num_units;
  int32_t group_heads;    // heads (dq) / key-value heads (dkdv) per scheduling group
  int32_t layout, causal;
  float scale_log2;       // |scale| * log2(e)
  float scale;
  int32_t neg_scale;      // scale < 0: S (S^T) is computed as -Q K^T (-K Q^T)
  const float* lse2;      // [B*H, S_q_pad]: lse * log2(e); +inf for rows >= S_q
  const float* dsum;      // [B*H, S_q_pad]: rowsum(dO * O); 0 for rows >= S_q
  uint32_t* err;
  uint64_t wait_limit_ns;
  // Element strides (batch, head, seq) of the tensors read or written
  // without a tensor map: O and dO by the row-statistics pass, dQ by the dQ
  // epilogue.  D is contiguous.
  int64_t o_st[3], do_st[3], dq_st[3];
};

template <int D>
struct Tile {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kChunks = D / 64;        // 128-byte column chunks of a 16-bit row
  static constexpr int kChunkBytes = 128 * 128; // one TMA box: 128 rows x 128 bytes
  static constexpr int kBytes = kChunks * kChunkBytes;
  static constexpr int kDSteps = D / 16;        // UMMA K steps over the head dim
};

// ---------------------------------------------------------------------------
// Small pieces shared by both kernels.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                         int layout, int32_t c0, int32_t s, int32_t h, int32_t b) {
  if (layout == 0)
    tma_load_4d(dst, map, bar, c0, s, h, b);
  else
    tma_load_4d(dst, map, bar, c0, h, s, b);
}

__device__ __forceinline__ void tma_store_tile(const CUtensorMap* map, uint32_t src, int layout,
                                               int32_t c0, int32_t s, int32_t h, int32_t b) {
  if (layout == 0)
    tma_store_4d(map, src, c0, s, h, b);
  else
    tma_store_4d(map, src, c0, h, s, b);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void mbar_wait_teardown(uint32_t bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit) return;
  }
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

template <int DT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return DT == kF16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}

__device__ __forceinline__ void st_global_v4(void* ptr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Epilogue helpers.  load_row: this thread's TMEM lane, D fp32 accumulator
// columns from `src` (one 32-column load at a time), times `mul`, rounded to
// 16-bit pairs; zeros with `zero`.  store_row: those D / 2 pairs to `dst`
// (2 * D contiguous bytes) with 16-byte stores.
template <int D, int DT>
__device__ __forceinline__ void load_row(uint32_t src, float mul, bool zero,
                                         uint32_t (&pk)[D / 2]) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t a[32];
    if (zero) {
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] = 0u;
    } else {
      tmem_ld_x32(src + 32 * c, a);
      tmem_wait_ld();
      reg_dep_x32(a);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[16 * c + i] = pack2<DT>(__uint_as_float(a[2 * i]) * mul, __uint_as_float(a[2 * i + 1]) * mul);
  }
}
template <int D>
__device__ __forceinline__ void store_row(uint8_t* dst, const uint32_t (&pk)[D / 2]) {
#pragma unroll
  for (int q = 0; q < D / 8; ++q)
    st_global_v4(dst + 16 * q, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}

// Ring position: slot index and the parity of its current use.
template <int NS>
struct Ring {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void advance() {
    if (++slot == NS) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Static persistent schedule (as the forward's): units in groups of
// `group_heads` heads; inside a group the longest units come first when
// causal and heads vary fastest; CTA `bid` takes unit w*grid + bid in even
// rounds and w*grid + grid-1-bid in odd rounds.
__device__ __forceinline__ int unit_of_round(int w, int grid, int bid) {
  return w * grid + ((w & 1) ? (grid - 1 - bid) : bid);
}

// unit -> (head index among `n_heads`, tile index among `n_tiles`); with
// `reverse` the tile order is descending (causal dq: the last query tile
// sees the most keys), else ascending (causal dkdv: the first key tile is
// seen by the most queries).
__device__ __forceinline__ void decode_unit(int u, int n_heads, int n_tiles, int group_heads,
                                            bool reverse, int& head, int& tile) {
  const int per_group = group_heads * n_tiles;
  const int g = u / per_group;
  const int r = u - g * per_group;
  const int heads = min(group_heads, n_heads - g * group_heads);
  const int rank = r / heads;
  head = g * group_heads + (r - rank * heads);
  tile = reverse ? (n_tiles - 1 - rank) : rank;
}

// Key/value blocks that query tile i needs.
__device__ __forceinline__ int dq_kv_blocks(const BwdParams& p, int i) {
  if (!p.causal) return p.n_kv_tiles;
  const int64_t last_row = min(static_cast<int64_t>(i) * 128 + 127, p.S_q - 1);
  const int64_t max_col = min(last_row, p.S_kv - 1);
  return static_cast<int>(max_col / 128) + 1;
}

// First query tile that sees key tile j (causal, top-left: key k is seen by
// queries q >= k): tile i sees it iff i*128 + 127 >= j*128, i.e. i >= j.
__device__ __forceinline__ int dkdv_first_q_tile(const BwdParams& p, int j) {
  return p.causal ? j : 0;
}

// ===========================================================================
// Preparation: lse2 = lse * log2(e) and dsum = rowsum(dO * O) per query row,
// padded to whole 128-row tiles (+inf / 0 past S_q).  D/8 threads per row,
// 16 bytes of O and dO each.
// ===========================================================================
template <int D, int DT>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const uint16_t* __restrict__ o,
                                                          const uint16_t* __restrict__ dout,
                                                          const float* __restrict__ lse,
                                                          BwdParams p, float* lse2, float* dsum) {
  constexpr int G = D / 8;
  const int64_t total = p.B * p.H * p.S_q_pad * G;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int sub = threadIdx.x % G;
  // The block iterates uniformly (base is the same for all its threads), so
  // every lane takes part in the shuffles below.
  // Row indices in 32 bits (a tensor of 2^32 rows of 16-bit elements would
  // not fit in device memory): the divisions are the loop's costliest work.
  const uint32_t s_q_pad = static_cast<uint32_t>(p.S_q_pad), n_h = static_cast<uint32_t>(p.H);
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x; base < total; base += stride) {
    const int64_t t = base + threadIdx.x;
    const bool active = t < total;
    const uint32_t row = active ? static_cast<uint32_t>(t / G) : 0u;  // (b*H + h) * S_q_pad + s
    const uint32_t bh = row / s_q_pad;
    const uint32_t s = row - bh * s_q_pad;
    float acc = 0.0f;
    if (active && s < p.S_q) {
      const int64_t b = bh / n_h, h = bh - static_cast<uint32_t>(b) * n_h;
      const int64_t off_o = b * p.o_st[0] + h * p.o_st[1] + s * p.o_st[2] + sub * 8;
      const int64_t off_do = b * p.do_st[0] + h * p.do_st[1] + s * p.do_st[2] + sub * 8;
      const uint4 ov = *reinterpret_cast<const uint4*>(o + off_o);
      const uint4 dv = *reinterpret_cast<const uint4*>(dout + off_do);
      const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
      const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float o0, o1, d0, d1;
        if (DT == kBF16) {
          o0 = __uint_as_float(ow[i] << 16);
          o1 = __uint_as_float(ow[i] & 0xFFFF0000u);
          d0 = __uint_as_float(dw[i] << 16);
          d1 = __uint_as_float(dw[i] & 0xFFFF0000u);
        } else {
          o0 = __half2float(__ushort_as_half(static_cast<unsigned short>(ow[i] & 0xFFFFu)));
          o1 = __half2float(__ushort_as_half(static_cast<unsigned short>(ow[i] >> 16)));
          d0 = __half2float(__ushort_as_half(static_cast<unsigned short>(dw[i] & 0xFFFFu)));
          d1 = __half2float(__ushort_as_half(static_cast<unsigned short>(dw[i] >> 16)));
        }
        acc = fmaf(o0, d0, acc);
        acc = fmaf(o1, d1, acc);
      }
    }
#pragma unroll
    for (int m = G / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m, G);
    if (active && sub == 0) {
      dsum[row] = acc;
      lse2[row] = (s < p.S_q) ? lse[static_cast<int64_t>(bh) * p.S_q + s] * 1.4426950408889634f
                              : CUDART_INF_F;
    }
  }
}

// ===========================================================================
// dQ kernel.
// ===========================================================================
// K and V stream through rings of their own: K_j is read by S_j and, a block
// later in time, by dQ += dS_j K_j, so K needs three slots for K_{j+1} to be
// in flight while K_{j-1} and K_j are still held; V_j is read by dP_j only.
template <int D>
struct DqCfg {
  using T = Tile<D>;
  static constexpr int kKSlots = T::kBytes >= 32768 ? 3 : 6;
  static constexpr int kVSlots = T::kBytes >= 32768 ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kDOOff = T::kBytes;
  static constexpr int kKOff = 2 * T::kBytes;
  static constexpr int kVOff = kKOff + kKSlots * T::kBytes;
  static constexpr int kBarOff = kVOff + kVSlots * T::kBytes;
  static constexpr int kNumBars = 2 * (kKSlots + kVSlots) + 11;
  static constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + 1024;
  static_assert(kSmem <= 232448, "shared memory budget");
  // Requested at launch: more than half of an SM's shared memory, so that
  // one CTA (and one 512-column TMEM allocation) runs per SM.
  static constexpr int kLaunchSmem = kSmem > 120 * 1024 ? kSmem : 120 * 1024;
  // TMEM columns: S, dP (128 fp32 each), dQ (D fp32), dS (64 packed 16-bit pairs).
  static constexpr uint32_t kS = 0, kDP = 128, kDQ = 256, kDS = 256 + D;
};

struct DqBars {
  uint32_t base;
  int nk, nv;
  __device__ uint32_t kfull(int s) const { return base + 8u * s; }
  __device__ uint32_t kempty(int s) const { return base + 8u * (nk + s); }
  __device__ uint32_t vfull(int s) const { return base + 8u * (2 * nk + s); }
  __device__ uint32_t vempty(int s) const { return base + 8u * (2 * nk + nv + s); }
  __device__ uint32_t x(int i) const { return base + 8u * (2 * (nk + nv) + i); }
  __device__ uint32_t q_full() const { return x(0); }
  __device__ uint32_t q_empty() const { return x(1); }
  __device__ uint32_t s_full() const { return x(2); }
  __device__ uint32_t s_free() const { return x(3); }
  __device__ uint32_t dp_full() const { return x(4); }
  __device__ uint32_t ds_ready() const { return x(5); }
  __device__ uint32_t dq_done() const { return x(6); }
  __device__ uint32_t dq_free() const { return x(7); }
  __device__ uint32_t drain() const { return x(8); }
  __device__ uint32_t do_full() const { return x(9); }
  __device__ uint32_t do_empty() const { return x(10); }
};

__device__ __forceinline__ void dq_decode(const BwdParams& p, int u, int& bh, int& i) {
  decode_unit(u, static_cast<int>(p.B * p.H), p.n_q_tiles, p.group_heads, p.causal != 0, bh, i);
}

// Producer: Q_i and dO_i once per unit, then K_0, V_0, K_1, V_1, ... into
// their rings.  Q and dO are reloaded as soon as the previous unit's last
// S and dP products have read them, so the next unit's loads overlap that
// unit's last block.
template <int D>
__device__ void dq_producer(const BwdParams& p, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                            const CUtensorMap* tmV, const CUtensorMap* tmDO, uint32_t smem,
                            const DqBars& bars, const WaitCtl& wc) {
  using C = DqCfg<D>;
  using T = Tile<D>;
  // The whole warp runs this role; one elected lane issues (see elect_one).
  const bool leader = elect_one();
  Ring<C::kKSlots> kr;
  Ring<C::kVSlots> vr;
  uint32_t k_issued = 0, v_issued = 0, it = 0, do_it = 0;
  bool ok = true;
  const int grid = gridDim.x, bid = blockIdx.x;
  for (int w = 0; ok; ++w) {
    const int u = unit_of_round(w, grid, bid);
    if (u >= p.num_units) break;
    int bh, i;
    dq_decode(p, u, bh, i);
    const int32_t b = static_cast<int32_t>(bh / p.H), h = static_cast<int32_t>(bh % p.H);
    const int32_t hk = h / p.kv_group;
    const int n = dq_kv_blocks(p, i);
    if (!mbar_wait(bars.q_empty(), (it & 1u) ^ 1u, wc)) { ok = false; break; }
    if (leader) mbar_arrive_expect_tx(bars.q_full(), T::kBytes);
    for (int c = 0; c < T::kChunks && leader; ++c)
      tma_tile(smem + C::kQOff + c * T::kChunkBytes, tmQ, bars.q_full(), p.layout, c * 64, i * 128,
               h, b);
    ++it;
    if (!mbar_wait(bars.do_empty(), (do_it & 1u) ^ 1u, wc)) { ok = false; break; }
    if (leader) mbar_arrive_expect_tx(bars.do_full(), T::kBytes);
    for (int c = 0; c < T::kChunks && leader; ++c)
      tma_tile(smem + C::kDOOff + c * T::kChunkBytes, tmDO, bars.do_full(), p.layout, c * 64,
               i * 128, h, b);
    ++do_it;
    for (int j = 0; j < n && ok; ++j) {
      if (!mbar_wait(bars.kempty(kr.slot), kr.phase ^ 1u, wc)) { ok = false; break; }
      if (leader) mbar_arrive_expect_tx(bars.kfull(kr.slot), T::kBytes);
      for (int c = 0; c < T::kChunks && leader; ++c)
        tma_tile(smem + C::kKOff + kr.slot * T::kBytes + c * T::kChunkBytes, tmK,
                 bars.kfull(kr.slot), p.layout, c * 64, j * 128, hk, b);
      kr.advance();
      ++k_issued;
      if (!mbar_wait(bars.vempty(vr.slot), vr.phase ^ 1u, wc)) { ok = false; break; }
      if (leader) mbar_arrive_expect_tx(bars.vfull(vr.slot), T::kBytes);
      for (int c = 0; c < T::kChunks && leader; ++c)
        tma_tile(smem + C::kVOff + vr.slot * T::kBytes + c * T::kChunkBytes, tmV,
                 bars.vfull(vr.slot), p.layout, c * 64, j * 128, hk, b);
      vr.advance();
      ++v_issued;
    }
  }
  if (!ok) {
    // Let loads already in flight land before the CTA's shared memory goes away.
    const uint32_t fk = k_issued > static_cast<uint32_t>(C::kKSlots) ? k_issued - C::kKSlots : 0u;
    for (uint32_t r = fk; r < k_issued; ++r)
      mbar_wait_teardown(bars.kfull(r % C::kKSlots), (r / C::kKSlots) & 1u, 20000000ull);
    const uint32_t fv = v_issued > static_cast<uint32_t>(C::kVSlots) ? v_issued - C::kVSlots : 0u;
    for (uint32_t r = fv; r < v_issued; ++r)
      mbar_wait_teardown(bars.vfull(r % C::kVSlots), (r / C::kVSlots) & 1u, 20000000ull);
    if (it > 0) mbar_wait_teardown(bars.q_full(), (it - 1) & 1u, 20000000ull);
    if (do_it > 0) mbar_wait_teardown(bars.do_full(), (do_it - 1) & 1u, 20000000ull);
  }
}

// K-major x K-major product over the head dim: D[128 x 128] = A[128 x D] B[128 x D]^T.
template <int D, int DT>
__device__ __forceinline__ void issue_ss(bool leader, uint32_t d_tmem, uint32_t a_lo,
                                         uint32_t b_lo, bool neg_b = false) {
  using T = Tile<D>;
  constexpr uint32_t hi = umma_desc_hi_sw128(1024);
  // neg_b: B negated (instruction descriptor bit 14), for S with a negative scale.
  const uint32_t idesc =
      umma_idesc(DT == kBF16 ? 1u : 0u, false, 128, 128) | (neg_b ? 1u << 14 : 0u);
#pragma unroll
  for (int kk = 0; kk < T::kDSteps; ++kk) {
    const uint32_t off =
        static_cast<uint32_t>(((kk * 32 / 128) * T::kChunkBytes + (kk * 32) % 128) >> 4);
    if (leader) umma_ss_w<false>(d_tmem, a_lo + off, hi, b_lo + off, hi, idesc, kk > 0 ? 1u : 0u);
  }
}

// D[128 x D] (+)= A[128 x 128] (TMEM, 16-bit pairs) B[128 x D] (rows of 128
// along K, MN-major).  A's K step kk (16 elements = 8 columns) sits at
// column a_col(kk).
template <int D, int DT, bool kSplitHalves>
__device__ __forceinline__ void issue_ts(bool leader, uint32_t d_tmem, uint32_t a_tmem,
                                         uint32_t b_lo, uint32_t accumulate) {
  constexpr uint32_t hi = umma_desc_hi_sw128(1024);
  constexpr uint32_t idesc = umma_idesc(DT == kBF16 ? 1u : 0u, true, 128, D);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t acol = kSplitHalves ? static_cast<uint32_t>(64 * (kk / 4) + 8 * (kk % 4))
                                       : static_cast<uint32_t>(8 * kk);
    const uint32_t off = static_cast<uint32_t>((kk * 16 * 128) >> 4);
    if (leader)
      umma_ts_w<false>(d_tmem, a_tmem + acol, b_lo + off, hi, idesc, kk > 0 ? 1u : accumulate);
  }
}

template <int D, int DT>
__device__ void dq_mma(const BwdParams& p, uint32_t tmem, uint32_t smem, const DqBars& bars,
                       const WaitCtl& wc) {
  // The whole warp runs this role; one elected lane issues (see elect_one).
  const bool leader = elect_one();
  using C = DqCfg<D>;
  using T = Tile<D>;
  constexpr uint32_t kTileW = T::kBytes >> 4;
  const uint32_t q_lo = umma_desc_lo(smem + C::kQOff, 16);
  const uint32_t do_lo = umma_desc_lo(smem + C::kDOOff, 16);
  const uint32_t k_kmaj0 = umma_desc_lo(smem + C::kKOff, 16);
  const uint32_t k_mn0 = umma_desc_lo(smem + C::kKOff, T::kChunkBytes);
  const uint32_t v_kmaj0 = umma_desc_lo(smem + C::kVOff, 16);
  const uint32_t tS = tmem + C::kS, tDP = tmem + C::kDP, tDQ = tmem + C::kDQ, tDS = tmem + C::kDS;
  Ring<C::kKSlots> kr;
  Ring<C::kVSlots> vr;
  uint32_t it = 0, s_issued = 0, ds_ph = 0, units = 0;
  bool ok = true;
  const int grid = gridDim.x, bid = blockIdx.x;
  for (int w = 0; ok; ++w) {
    const int u = unit_of_round(w, grid, bid);
    if (u >= p.num_units) break;
    int bh, i;
    dq_decode(p, u, bh, i);
    const int n = dq_kv_blocks(p, i);
    if (!mbar_wait(bars.q_full(), it & 1u, wc)) { ok = false; break; }
    // S_0 = Q K_0^T once the softmax warps have read the previous S.
    int slotK = kr.slot;
    if (!mbar_wait(bars.kfull(slotK), kr.phase, wc)) { ok = false; break; }
    kr.advance();
    if (s_issued > 0 && !mbar_wait(bars.s_free(), (s_issued - 1) & 1u, wc)) { ok = false; break; }
    tc_fence_after();
    issue_ss<D, DT>(leader, tS, q_lo, k_kmaj0 + slotK * kTileW, p.neg_scale != 0);
    umma_commit_if(leader, bars.s_full());
    ++s_issued;
    // Q and dO go back to the producer once the unit's last S and dP
    // products (the commit covers every earlier product) have read them.
    if (n == 1) umma_commit_if(leader, bars.q_empty());
    // dP_0 = dO V_0^T.
    {
      if (!mbar_wait(bars.do_full(), it & 1u, wc)) { ok = false; break; }
      const int slotV = vr.slot;
      if (!mbar_wait(bars.vfull(slotV), vr.phase, wc)) { ok = false; break; }
      vr.advance();
      tc_fence_after();
      issue_ss<D, DT>(leader, tDP, do_lo, v_kmaj0 + slotV * kTileW);
      umma_commit_if(leader, bars.dp_full());
      umma_commit_if(leader, bars.vempty(slotV));
      if (n == 1) umma_commit_if(leader, bars.do_empty());
    }
    ++it;
    for (int j = 0; j < n; ++j) {
      const bool has_next = j + 1 < n;
      int slotKn = slotK;
      // The barriers of this block, probed together without blocking (this
      // warp's issue sets the pace; a blocking wait costs it about a product):
      // bit 0 K_{j+1} loaded, 1 S read, 2 dS_j written, 3 V_{j+1} loaded.
      const uint32_t done = (mbar_test_wait(bars.kfull(kr.slot), kr.phase) ? 1u : 0u) |
                            (mbar_test_wait(bars.s_free(), (s_issued - 1) & 1u) ? 2u : 0u) |
                            (mbar_test_wait(bars.ds_ready(), ds_ph) ? 4u : 0u) |
                            (mbar_test_wait(bars.vfull(vr.slot), vr.phase) ? 8u : 0u);
      if (has_next) {
        slotKn = kr.slot;
        if (!(done & 1u) && !mbar_wait(bars.kfull(slotKn), kr.phase, wc)) { ok = false; break; }
        kr.advance();
        if (!(done & 2u) && !mbar_wait(bars.s_free(), (s_issued - 1) & 1u, wc)) { ok = false; break; }
        tc_fence_after();
        issue_ss<D, DT>(leader, tS, q_lo, k_kmaj0 + slotKn * kTileW, p.neg_scale != 0);
        umma_commit_if(leader, bars.s_full());
        ++s_issued;
        if (j + 2 == n) umma_commit_if(leader, bars.q_empty());
      }
      // dQ (+)= dS_j K_j once dS_j is in TMEM; the first product of a unit
      // overwrites dQ, after the previous unit's epilogue has read it.
      if (!(done & 4u) && !mbar_wait(bars.ds_ready(), ds_ph, wc)) { ok = false; break; }
      ds_ph ^= 1u;
      if (j == 0 && units > 0 && !mbar_wait(bars.dq_free(), (units - 1) & 1u, wc)) { ok = false; break; }
      tc_fence_after();
      issue_ts<D, DT, false>(leader, tDQ, tDS, k_mn0 + slotK * kTileW, j > 0 ? 1u : 0u);
      umma_commit_if(leader, bars.kempty(slotK));
      if (has_next) {
        const int slotV = vr.slot;
        if (!(done & 8u) && !mbar_wait(bars.vfull(slotV), vr.phase, wc)) { ok = false; break; }
        vr.advance();
        tc_fence_after();
        issue_ss<D, DT>(leader, tDP, do_lo, v_kmaj0 + slotV * kTileW);
        umma_commit_if(leader, bars.dp_full());
        umma_commit_if(leader, bars.vempty(slotV));
        if (j + 2 == n) umma_commit_if(leader, bars.do_empty());
      }
      slotK = slotKn;
    }
    if (!ok) break;
    umma_commit_if(leader, bars.dq_done());
    ++units;
  }
  umma_commit_if(leader, bars.drain());
  mbar_wait_teardown(bars.drain(), 0u, ok ? 2000000000ull : 20000000ull);
}

// Packed fp32 pair product (sm_100+), beside the pair FMA / add of fa_ptx.cuh:
// the P and dS arithmetic of the backward's softmax warps runs on pairs.
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

template <int D, int DT>
__device__ void dq_softmax(const BwdParams& p, uint32_t tmem, int warp, int lane,
                           const DqBars& bars, const WaitCtl& wc) {
  using C = DqCfg<D>;
  const int quad = warp & 3, half = warp >> 2;
  const int r = quad * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t tS = tmem + lane_off + C::kS + 64 * half;
  const uint32_t tDP = tmem + lane_off + C::kDP + 64 * half;
  const uint32_t tDS = tmem + lane_off + C::kDS + 32 * half;
  // A masked score is -inf and must give p = 0: keep the scale positive.
  const float sl2 = fmaxf(p.scale_log2, 1e-30f);
  uint32_t s_ph = 0, dp_ph = 0;
  const int grid = gridDim.x, bid = blockIdx.x;
  for (int w = 0;; ++w) {
    const int u = unit_of_round(w, grid, bid);
    if (u >= p.num_units) break;
    int bh, i;
    dq_decode(p, u, bh, i);
    const int n = dq_kv_blocks(p, i);
    const int64_t qi = static_cast<int64_t>(i) * 128 + r;
    const float neg_lse2 = -p.lse2[bh * p.S_q_pad + qi];
    const float dsum = p.dsum[bh * p.S_q_pad + qi];
    const int64_t col_end = p.causal ? min(qi + 1, p.S_kv) : p.S_kv;  // keys < col_end visible
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait(bars.s_full(), s_ph, wc)) { ok = false; break; }
      s_ph ^= 1u;
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld_x32(tS, sr[0]);
      tmem_ld_x32(tS + 32, sr[1]);
      tmem_wait_ld();
      reg_dep_x32(sr[0]);
      reg_dep_x32(sr[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.s_free());
      const int64_t col0 = static_cast<int64_t>(j) * 128 + 64 * half;
      const bool masked = (static_cast<int64_t>(j) * 128 + 128 > p.S_kv) ||
                          (p.causal && static_cast<int64_t>(j) * 128 + 127 > static_cast<int64_t>(i) * 128);
      const int lim = static_cast<int>(max(min(col_end - col0, int64_t(64)), int64_t(0)));
      // Two straight-line loops, the mask test outside them (a block-uniform
      // branch inside the unrolled loop splits it into basic blocks).
      float pr[64];
      const uint64_t sl2x2 = f2_pack(sl2, sl2), nlse2 = f2_pack(neg_lse2, neg_lse2);
      if (masked) {
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float x0 = (c < lim) ? __uint_as_float(sr[c >> 5][c & 31]) : -CUDART_INF_F;
          const float x1 =
              (c + 1 < lim) ? __uint_as_float(sr[c >> 5][(c + 1) & 31]) : -CUDART_INF_F;
          f2_unpack(f2_fma(f2_pack(x0, x1), sl2x2, nlse2), pr[c], pr[c + 1]);
          pr[c] = ex2(pr[c]);
          pr[c + 1] = ex2(pr[c + 1]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c >> 5][c & 31]),
                                   __uint_as_float(sr[c >> 5][(c + 1) & 31])),
                           sl2x2, nlse2),
                    pr[c], pr[c + 1]);
          pr[c] = ex2(pr[c]);
          pr[c + 1] = ex2(pr[c + 1]);
        }
      }
      if (!mbar_wait(bars.dp_full(), dp_ph, wc)) { ok = false; break; }
      dp_ph ^= 1u;
      tc_fence_after();
      uint32_t dr[2][32];
      tmem_ld_x32(tDP, dr[0]);
      tmem_ld_x32(tDP + 32, dr[1]);
      tmem_wait_ld();
      reg_dep_x32(dr[0]);
      reg_dep_x32(dr[1]);
      uint32_t pk[32];
      const uint64_t ndsum2 = f2_pack(-dsum, -dsum);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float d0, d1;
        f2_unpack(f2_mul(f2_pack(pr[2 * c], pr[2 * c + 1]),
                         f2_add(f2_pack(__uint_as_float(dr[(2 * c) >> 5][(2 * c) & 31]),
                                        __uint_as_float(dr[(2 * c + 1) >> 5][(2 * c + 1) & 31])),
                                ndsum2)),
                  d0, d1);
        pk[c] = pack2<DT>(d0, d1);
      }
      tmem_st_x32(tDS, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.ds_ready());
    }
    if (!ok) break;
  }
}

// dQ epilogue (warps 12-15, one TMEM lane quarter each): once a unit's last
// product is done, dQ = scale * (dS K) is read out of TMEM and handed back
// to the issuing warp, then written as 16-bit, one row per thread with
// 16-byte stores (rows past S_q are not written).
template <int D, int DT>
__device__ void dq_epilogue(const BwdParams& p, void* dq_out, uint32_t tmem, int warp, int lane,
                            const DqBars& bars, const WaitCtl& wc) {
  using C = DqCfg<D>;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const uint32_t tDQ = tmem + (static_cast<uint32_t>(quad * 32) << 16) + C::kDQ;
  uint32_t dq_ph = 0;
  const int grid = gridDim.x, bid = blockIdx.x;
  for (int w = 0;; ++w) {
    const int u = unit_of_round(w, grid, bid);
    if (u >= p.num_units) break;
    int bh, i;
    dq_decode(p, u, bh, i);
    const int64_t qi = static_cast<int64_t>(i) * 128 + r;
    if (!mbar_wait(bars.dq_done(), dq_ph, wc)) break;
    dq_ph ^= 1u;
    tc_fence_after();
    uint32_t pk[D / 2];
    load_row<D, DT>(tDQ, p.scale, false, pk);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.dq_free());
    if (qi < p.S_q) {
      const int64_t b = bh / p.H, h = bh - b * p.H;
      store_row<D>(static_cast<uint8_t*>(dq_out) +
                       (b * p.dq_st[0] + h * p.dq_st[1] + qi * p.dq_st[2]) * 2,
                   pk);
    }
  }
}

template <int D, int DT>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                     void* dq_out, const __grid_constant__ BwdParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const DqBars bars{base + static_cast<uint32_t>(C::kBarOff), C::kKSlots, C::kVSlots};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBarOff + C::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kKSlots; ++s) {
      mbar_init(bars.kfull(s), 1);
      mbar_init(bars.kempty(s), 1);
    }
    for (int s = 0; s < C::kVSlots; ++s) {
      mbar_init(bars.vfull(s), 1);
      mbar_init(bars.vempty(s), 1);
    }
    mbar_init(bars.q_full(), 1);
    mbar_init(bars.q_empty(), 1);
    mbar_init(bars.do_full(), 1);
    mbar_init(bars.do_empty(), 1);
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.s_free(), 8);
    mbar_init(bars.dp_full(), 1);
    mbar_init(bars.ds_ready(), 8);
    mbar_init(bars.dq_done(), 1);
    mbar_init(bars.dq_free(), 4);
    mbar_init(bars.drain(), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{p.wait_limit_ns, p.err, abort_flag};
  // Launched as a programmatic dependent of the row-statistics pass: wait for
  // it before any global access, then let the dK/dV kernel (which needs only
  // that pass) take the SMs this grid leaves as its CTAs finish.
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  if (warp < kProducerWarp) {
    reg_alloc_inc<kRegSoftmax>();
    dq_softmax<D, DT>(p, tmem, warp, lane, bars, wc);
  } else if (warp < kEpiWarp0) {
    reg_alloc_dec<kRegControl>();
    if (warp == kProducerWarp)
      dq_producer<D>(p, &tmQ, &tmK, &tmV, &tmDO, base, bars, wc);
    else if (warp == kMmaWarp)
      dq_mma<D, DT>(p, tmem, base, bars, wc);
  } else {
    reg_alloc_dec<kRegEpilogue>();
    dq_epilogue<D, DT>(p, dq_out, tmem, warp, lane, bars, wc);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ===========================================================================
// dK / dV kernel.
// ===========================================================================
template <int D>
struct KvCfg {
  using T = Tile<D>;
  static constexpr int kStages = 2;
  static constexpr int kStageBytes = 2 * T::kBytes + 1024;  // Q_i, dO_i, lse2[128], dsum[128]
  static constexpr int kKOff = 0;
  static constexpr int kVOff = T::kBytes;
  static constexpr int kRingOff = 2 * T::kBytes;
  // Epilogue staging: per epilogue warp 16 rows x 2 * D bytes, as 128-byte
  // swizzled boxes of 16 rows x 128 bytes (one per 64 columns).
  static constexpr int kEpiOff = kRingOff + kStages * kStageBytes;
  static constexpr int kEpiWarpBytes = 16 * 2 * D;
  static constexpr int kBarOff = kEpiOff + 4 * kEpiWarpBytes;
  static constexpr int kNumBars = 2 * kStages + 10;
  static constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + 1024;
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static constexpr int kLaunchSmem = kSmem > 120 * 1024 ? kSmem : 120 * 1024;
  // TMEM columns: S^T, dP^T (128 fp32 each), dV, dK (D fp32 each).  P^T and
  // dS^T (16-bit pairs) overwrite the first 32 columns of each 64-column half
  // of S^T and dP^T.
  static constexpr uint32_t kS = 0, kDP = 128, kDV = 256, kDK = 256 + D;
};

struct KvBars {
  uint32_t base;
  __device__ uint32_t full(int s) const { return base + 8u * s; }
  __device__ uint32_t empty(int s) const { return base + 8u * (2 + s); }
  __device__ uint32_t kv_full() const { return base + 8u * 4; }
  __device__ uint32_t dv_free() const { return base + 8u * 5; }  // dV read by the epilogue
  __device__ uint32_t s_full() const { return base + 8u * 6; }
  __device__ uint32_t p_ready() const { return base + 8u * 7; }
  __device__ uint32_t dp_full() const { return base + 8u * 8; }
  __device__ uint32_t ds_ready() const { return base + 8u * 9; }
  __device__ uint32_t dkv_done() const { return base + 8u * 10; }
  __device__ uint32_t drain() const { return base + 8u * 11; }
  __device__ uint32_t kv_empty() const { return base + 8u * 12; }  // K, V read by their last products
  __device__ uint32_t dk_free() const { return base + 8u * 13; }   // dK read by the epilogue
};

struct KvUnit {
  int b, hk, j;   // batch, key/value head, key tile
  int i0, n_i;    // query tiles [i0, i0 + n_i) of each query head of the group
  int n_steps;    // kv_group * n_i
};

__device__ __forceinline__ KvUnit kv_decode(const BwdParams& p, int u) {
  KvUnit k;
  int bhk, j;
  decode_unit(u, static_cast<int>(p.B * p.H_kv), p.n_kv_tiles, p.group_heads, false, bhk, j);
  k.b = static_cast<int>(bhk / p.H_kv);
  k.hk = static_cast<int>(bhk % p.H_kv);
  k.j = j;
  k.i0 = dkdv_first_q_tile(p, j);
  k.n_i = max(0, p.n_q_tiles - k.i0);
  k.n_steps = p.kv_group * k.n_i;
  return k;
}

__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

template <int D>
__device__ void kv_producer(const BwdParams& p, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                            const CUtensorMap* tmV, const CUtensorMap* tmDO, uint32_t smem,
                            const KvBars& bars, const WaitCtl& wc) {
  using C = KvCfg<D>;
  using T = Tile<D>;
  // The whole warp runs this role; one elected lane issues (see elect_one).
  const bool leader = elect_one();
  Ring<C::kStages> ring;
  uint32_t issued = 0, kv_loads = 0;
  bool ok = true;
  const int grid = gridDim.x, bid = blockIdx.x;
  for (int w = 0; ok; ++w) {
    const int u = unit_of_round(w, grid, bid);
    if (u >= p.num_units) break;
    const KvUnit k = kv_decode(p, u);
    if (k.n_steps == 0) continue;
    // The previous K / V tiles are reloaded once that unit's last S^T and
    // dP^T products have read them: the load overlaps its last step.
    if (kv_loads > 0 && !mbar_wait(bars.kv_empty(), (kv_loads - 1) & 1u, wc)) { ok = false; break; }
    if (leader) mbar_arrive_expect_tx(bars.kv_full(), 2 * T::kBytes);
    for (int c = 0; c < T::kChunks && leader; ++c) {
      tma_tile(smem + C::kKOff + c * T::kChunkBytes, tmK, bars.kv_full(), p.layout, c * 64,
               k.j * 128, k.hk, k.b);
      tma_tile(smem + C::kVOff + c * T::kChunkBytes, tmV, bars.kv_full(), p.layout, c * 64,
               k.j * 128, k.hk, k.b);
    }
    ++kv_loads;
    for (int s = 0; s < k.n_steps && ok; ++s) {
      const int hl = s / k.n_i;
      const int i = k.i0 + (s - hl * k.n_i);
      const int h = k.hk * p.kv_group + hl;
      if (!mbar_wait(bars.empty(ring.slot), ring.phase ^ 1u, wc)) { ok = false; break; }
      const uint32_t st = smem + C::kRingOff + ring.slot * C::kStageBytes;
      const uint32_t bar = bars.full(ring.slot);
      if (leader) mbar_arrive_expect_tx(bar, 2 * T::kBytes + 1024);
      for (int c = 0; c < T::kChunks && leader; ++c) {
        tma_tile(st + c * T::kChunkBytes, tmQ, bar, p.layout, c * 64, i * 128, h, k.b);
        tma_tile(st + T::kBytes + c * T::kChunkBytes, tmDO, bar, p.layout, c * 64, i * 128, h,
                 k.b);
      }
      const int64_t row = (static_cast<int64_t>(k.b) * p.H + h) * p.S_q_pad + static_cast<int64_t>(i) * 128;
      if (leader) {
        bulk_load_1d(st + 2 * T::kBytes, p.lse2 + row, 512, bar);
        bulk_load_1d(st + 2 * T::kBytes + 512, p.dsum + row, 512, bar);
      }
      ring.advance();
      ++issued;
    }
  }
  if (!ok) {
    const uint32_t first = issued > static_cast<uint32_t>(C::kStages) ? issued - C::kStages : 0u;
    for (uint32_t r = first; r < issued; ++r)
      mbar_wait_teardown(bars.full(r % C::kStages), (r / C::kStages) & 1u, 20000000ull);
    if (kv_loads > 0) mbar_wait_teardown(bars.kv_full(), (kv_loads - 1) & 1u, 20000000ull);
  }
}

template <int D, int DT>
__device__ void kv_mma(const BwdParams& p, uint32_t tmem, uint32_t smem, const KvBars& bars,
                       const WaitCtl& wc) {
  // The whole warp runs this role; one elected lane issues (see elect_one).
  const bool leader = elect_one();
  using C = KvCfg<D>;
  using T = Tile<D>;
  constexpr uint32_t kStageW = C::kStageBytes >> 4;
  constexpr uint32_t kTileW = T::kBytes >> 4;
  const uint32_t k_lo = umma_desc_lo(smem + C::kKOff, 16);
  const uint32_t v_lo = umma_desc_lo(smem + C::kVOff, 16);
  const uint32_t q_kmaj0 = umma_desc_lo(smem + C::kRingOff, 16);
  const uint32_t q_mn0 = umma_desc_lo(smem + C::kRingOff, T::kChunkBytes);
  const uint32_t tS = tmem + C::kS, tDP = tmem + C::kDP, tDV = tmem + C::kDV, tDK = tmem + C::kDK;
  Ring<C::kStages> ring;
  uint32_t kv_loads = 0, p_ph = 0, ds_ph = 0, units = 0;
  bool ok = true;
  const int grid = gridDim.x, bid = blockIdx.x;
  for (int w = 0; ok; ++w) {
    const int u = unit_of_round(w, grid, bid);
    if (u >= p.num_units) break;
    const KvUnit k = kv_decode(p, u);
    // The previous unit's epilogue must have read dV (dK) from TMEM before
    // this unit's first dV (dK) product overwrites it -- and both before this
    // unit's dkv_done, so that its phases never run two ahead of the epilogue.
    const bool acc_wait = units > 0;
    const uint32_t acc_ph = (units - 1u) & 1u;
    ++units;
    if (k.n_steps == 0) {
      if (acc_wait && (!mbar_wait(bars.dv_free(), acc_ph, wc) ||
                       !mbar_wait(bars.dk_free(), acc_ph, wc))) { ok = false; break; }
      umma_commit_if(leader, bars.dkv_done());  // nothing to accumulate: dK = dV = 0
      continue;
    }
    if (!mbar_wait(bars.kv_full(), kv_loads & 1u, wc)) { ok = false; break; }
    ++kv_loads;
    int st = ring.slot;
    if (!mbar_wait(bars.full(st), ring.phase, wc)) { ok = false; break; }
    ring.advance();
    tc_fence_after();
    issue_ss<D, DT>(leader, tS, k_lo, q_kmaj0 + st * kStageW, p.neg_scale != 0);
    umma_commit_if(leader, bars.s_full());
    issue_ss<D, DT>(leader, tDP, v_lo, q_kmaj0 + st * kStageW + kTileW);
    umma_commit_if(leader, bars.dp_full());
    // K and V go back to the producer after the unit's last S^T and dP^T
    // (the commit covers every earlier product).
    if (k.n_steps == 1) umma_commit_if(leader, bars.kv_empty());
    for (int s = 0; s < k.n_steps; ++s) {
      const bool has_next = s + 1 < k.n_steps;
      // Probed together without blocking: bit 0 P^T written, 1 the next
      // query tile loaded, 2 dS^T written.
      const uint32_t done = (mbar_test_wait(bars.p_ready(), p_ph) ? 1u : 0u) |
                            (mbar_test_wait(bars.full(ring.slot), ring.phase) ? 2u : 0u) |
                            (mbar_test_wait(bars.ds_ready(), ds_ph) ? 4u : 0u);
      // dV (+)= P^T dO_s.
      if (!(done & 1u) && !mbar_wait(bars.p_ready(), p_ph, wc)) { ok = false; break; }
      p_ph ^= 1u;
      if (s == 0 && acc_wait && !mbar_wait(bars.dv_free(), acc_ph, wc)) { ok = false; break; }
      tc_fence_after();
      issue_ts<D, DT, true>(leader, tDV, tS, q_mn0 + st * kStageW + kTileW, s > 0 ? 1u : 0u);
      int st_n = st;
      if (has_next) {
        st_n = ring.slot;
        if (!(done & 2u) && !mbar_wait(bars.full(st_n), ring.phase, wc)) { ok = false; break; }
        ring.advance();
        tc_fence_after();
        issue_ss<D, DT>(leader, tS, k_lo, q_kmaj0 + st_n * kStageW, p.neg_scale != 0);
        umma_commit_if(leader, bars.s_full());
      }
      // dK (+)= dS^T Q_s.
      if (!(done & 4u) && !mbar_wait(bars.ds_ready(), ds_ph, wc)) { ok = false; break; }
      ds_ph ^= 1u;
      if (s == 0 && acc_wait && !mbar_wait(bars.dk_free(), acc_ph, wc)) { ok = false; break; }
      tc_fence_after();
      issue_ts<D, DT, true>(leader, tDK, tDP, q_mn0 + st * kStageW, s > 0 ? 1u : 0u);
      umma_commit_if(leader, bars.empty(st));
      if (has_next) {
        issue_ss<D, DT>(leader, tDP, v_lo, q_kmaj0 + st_n * kStageW + kTileW);
        umma_commit_if(leader, bars.dp_full());
        if (s + 2 == k.n_steps) umma_commit_if(leader, bars.kv_empty());
      }
      st = st_n;
    }
    if (!ok) break;
    umma_commit_if(leader, bars.dkv_done());
  }
  umma_commit_if(leader, bars.drain());
  mbar_wait_teardown(bars.drain(), 0u, ok ? 2000000000ull : 20000000ull);
}

template <int D, int DT>
__device__ void kv_softmax(const BwdParams& p, uint32_t tmem, uint32_t smem, int warp, int lane,
                           const KvBars& bars, const WaitCtl& wc) {
  using C = KvCfg<D>;
  const int quad = warp & 3, half = warp >> 2;
  const int r = quad * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t tS = tmem + lane_off + C::kS + 64 * half;
  const uint32_t tDP = tmem + lane_off + C::kDP + 64 * half;
  const uint32_t tDV = tmem + lane_off + C::kDV;
  const uint32_t tDK = tmem + lane_off + C::kDK;
  const float sl2 = fmaxf(p.scale_log2, 1e-30f);
  uint32_t s_ph = 0, dp_ph = 0;
  Ring<C::kStages> ring;
  const int grid = gridDim.x, bid = blockIdx.x;
  for (int w = 0;; ++w) {
    const int u = unit_of_round(w, grid, bid);
    if (u >= p.num_units) break;
    const KvUnit k = kv_decode(p, u);
    const int64_t kj = static_cast<int64_t>(k.j) * 128 + r;
    const bool key_valid = kj < p.S_kv;
    bool ok = true;
    for (int s = 0; s < k.n_steps; ++s) {
      const int hl = s / k.n_i;
      const int i = k.i0 + (s - hl * k.n_i);
      const uint32_t st = smem + C::kRingOff + ring.slot * C::kStageBytes;
      const uint32_t sLse = st + 2 * Tile<D>::kBytes + 4 * 64 * half;
      const uint32_t sDsum = sLse + 512;
      const uint32_t st_bar = bars.full(ring.slot), st_ph = ring.phase;
      ring.advance();
      // Query q = i*128 + 64*half + c is visible to key kj iff q >= kj
      // (causal) and kj < S_kv; queries past S_q have lse2 = +inf (p = 0).
      // Only the diagonal tile (i == j) and the last key tile need a mask.
      const int64_t q0 = static_cast<int64_t>(i) * 128 + 64 * half;
      const bool masked = (p.causal && i == k.j) || (static_cast<int64_t>(k.j) * 128 + 128 > p.S_kv);
      const int lo = !key_valid ? 64
                     : p.causal ? static_cast<int>(max(min(kj - q0, int64_t(64)), int64_t(0)))
                                : 0;
      // The stage's lse2 / dsum arrived with its Q / dO tiles.
      if (!mbar_wait(st_bar, st_ph, wc)) { ok = false; break; }
      if (!mbar_wait(bars.s_full(), s_ph, wc)) { ok = false; break; }
      s_ph ^= 1u;
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld_x32(tS, sr[0]);
      tmem_ld_x32(tS + 32, sr[1]);
      tmem_wait_ld();
      reg_dep_x32(sr[0]);
      reg_dep_x32(sr[1]);
      // Two straight-line loops, the mask test outside them (as in dq_softmax).
      float pr[64];
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      if (masked) {
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l4 = ld_shared_f4(sLse + 16 * c4);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int c = 4 * c4 + e;
            const float x0 = (c >= lo) ? __uint_as_float(sr[c >> 5][c & 31]) : -CUDART_INF_F;
            const float x1 =
                (c + 1 >= lo) ? __uint_as_float(sr[c >> 5][(c + 1) & 31]) : -CUDART_INF_F;
            f2_unpack(f2_fma(f2_pack(x0, x1), sl2x2, f2_pack(-lv[e], -lv[e + 1])), pr[c],
                      pr[c + 1]);
            pr[c] = ex2(pr[c]);
            pr[c + 1] = ex2(pr[c + 1]);
          }
        }
      } else {
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l4 = ld_shared_f4(sLse + 16 * c4);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int c = 4 * c4 + e;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c >> 5][c & 31]),
                                     __uint_as_float(sr[c >> 5][(c + 1) & 31])),
                             sl2x2, f2_pack(-lv[e], -lv[e + 1])),
                      pr[c], pr[c + 1]);
            pr[c] = ex2(pr[c]);
            pr[c + 1] = ex2(pr[c + 1]);
          }
        }
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = pack2<DT>(pr[2 * c], pr[2 * c + 1]);
        tmem_st_x32(tS, pk);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.p_ready());
      if (!mbar_wait(bars.dp_full(), dp_ph, wc)) { ok = false; break; }
      dp_ph ^= 1u;
      tc_fence_after();
      uint32_t dr[2][32];
      tmem_ld_x32(tDP, dr[0]);
      tmem_ld_x32(tDP + 32, dr[1]);
      tmem_wait_ld();
      reg_dep_x32(dr[0]);
      reg_dep_x32(dr[1]);
      {
        uint32_t pk[32];
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 d4 = ld_shared_f4(sDsum + 16 * c4);
          const int c = 4 * c4;
          float a0, a1, a2, a3;
          f2_unpack(f2_mul(f2_pack(pr[c], pr[c + 1]),
                           f2_add(f2_pack(__uint_as_float(dr[c >> 5][c & 31]),
                                          __uint_as_float(dr[c >> 5][(c + 1) & 31])),
                                  f2_pack(-d4.x, -d4.y))),
                    a0, a1);
          f2_unpack(f2_mul(f2_pack(pr[c + 2], pr[c + 3]),
                           f2_add(f2_pack(__uint_as_float(dr[c >> 5][(c + 2) & 31]),
                                          __uint_as_float(dr[c >> 5][(c + 3) & 31])),
                                  f2_pack(-d4.z, -d4.w))),
                    a2, a3);
          pk[2 * c4] = pack2<DT>(a0, a1);
          pk[2 * c4 + 1] = pack2<DT>(a2, a3);
        }
        tmem_st_x32(tDP, pk);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.ds_ready());
    }
    if (!ok) break;
  }
}

// dK / dV epilogue (warps 12-15, one TMEM lane quarter each): once a unit's
// last product is done, dV, then dK = scale * (dS^T Q), is read out of TMEM,
// handed back to the issuing warp (the next unit's first dV / dK product
// overwrites it) and rounded to 16-bit; each warp then stages its 32 key rows
// in two rounds of 16 in shared memory and writes them by TMA stores, which
// clip rows past S_kv (the tensor cores, reading their operands from the same
// shared memory, lose far less to these than to per-thread row stores).  A
// key tile that no query sees writes zeros.
template <int D, int DT>
__device__ void kv_epilogue(const BwdParams& p, const CUtensorMap* tmDK, const CUtensorMap* tmDV,
                            uint32_t tmem, uint32_t smem, int warp, int lane, const KvBars& bars,
                            const WaitCtl& wc) {
  using C = KvCfg<D>;
  // Issues this warp's bulk stores and waits for them (a bulk async-group
  // belongs to the thread that committed it; see elect_one).
  const bool leader = elect_one();
  const int quad = warp & 3;
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t stage = smem + C::kEpiOff + static_cast<uint32_t>(quad * C::kEpiWarpBytes);
  uint32_t done_ph = 0;
  const int grid = gridDim.x, bid = blockIdx.x;
  for (int w = 0;; ++w) {
    const int u = unit_of_round(w, grid, bid);
    if (u >= p.num_units) break;
    const KvUnit k = kv_decode(p, u);
    if (!mbar_wait(bars.dkv_done(), done_ph, wc)) break;
    done_ph ^= 1u;
    tc_fence_after();
    const bool zero = k.n_steps == 0;
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {  // dV, then dK
      uint32_t pk[D / 2];
      load_row<D, DT>(tmem + lane_off + (which ? C::kDK : C::kDV), which ? p.scale : 1.0f, zero,
                      pk);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(which ? bars.dk_free() : bars.dv_free());
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        // The previous stores from the staging boxes must have read them.
        if (leader) bulk_wait_group_read0();
        __syncwarp();
        if ((lane >> 4) == rr) {
          const int rl = lane & 15;
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              st_shared_v4(stage + h * 2048 + rl * 128 + ((c ^ (rl & 7)) << 4), pk[32 * h + 4 * c],
                           pk[32 * h + 4 * c + 1], pk[32 * h + 4 * c + 2], pk[32 * h + 4 * c + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int32_t row = k.j * 128 + quad * 32 + 16 * rr;
        if (leader && row < p.S_kv) {
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_store_tile(which ? tmDK : tmDV, stage + h * 2048, p.layout, 64 * h, row, k.hk, k.b);
          bulk_commit_group();
        }
      }
    }
  }
  if (leader) bulk_wait_group0();
  __syncwarp();
}

template <int D, int DT>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
                       const __grid_constant__ BwdParams p) {
  using C = KvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const KvBars bars{base + static_cast<uint32_t>(C::kBarOff)};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBarOff + C::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    mbar_init(bars.kv_full(), 1);
    mbar_init(bars.dv_free(), 4);
    mbar_init(bars.dk_free(), 4);
    mbar_init(bars.kv_empty(), 1);
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.p_ready(), 8);
    mbar_init(bars.dp_full(), 1);
    mbar_init(bars.ds_ready(), 8);
    mbar_init(bars.dkv_done(), 1);
    mbar_init(bars.drain(), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmDK);
    tma_prefetch_desc(&tmDV);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{p.wait_limit_ns, p.err, abort_flag};
  // Launched as a programmatic dependent of the dQ kernel, which it does not
  // read (both read only the inputs and the row statistics, complete before
  // the dQ kernel let this grid start): no wait before the work.  But this
  // grid finishes only after the dQ kernel has, so that work queued after the
  // backward on the stream sees dQ too.
  if (warp < kProducerWarp) {
    reg_alloc_inc<kRegSoftmax>();
    kv_softmax<D, DT>(p, tmem, base, warp, lane, bars, wc);
  } else if (warp < kEpiWarp0) {
    reg_alloc_dec<kRegControl>();
    if (warp == kProducerWarp)
      kv_producer<D>(p, &tmQ, &tmK, &tmV, &tmDO, base, bars, wc);
    else if (warp == kMmaWarp)
      kv_mma<D, DT>(p, tmem, base, bars, wc);
  } else {
    reg_alloc_dec<kRegEpilogue>();
    kv_epilogue<D, DT>(p, &tmDK, &tmDV, tmem, base, warp, lane, bars, wc);
  }
  griddep_wait();
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Host-side launchers (explicit instantiations in fa_bwd_inst_*.cu).
template <int D, int DT>
cudaError_t launch_fa_bwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& dout, void* dq_ptr, const CUtensorMap& dk,
                          const CUtensorMap& dv, const void* o, const void* dout_ptr,
                          const float* lse, float* lse2, float* dsum, const BwdParams& p_dq,
                          const BwdParams& p_kv, int grid_dq, int grid_kv, int grid_prep,
                          cudaStream_t stream) {
  // Every launch reports its own status (cudaLaunchKernelEx), so an error
  // left pending by other code on this thread is never taken for ours.  The
  // dQ and dK/dV kernels are programmatic dependents of the launch before
  // them (see their kernels for the waits).
  cudaError_t e;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_prep);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    e = cudaLaunchKernelEx(&cfg, fa_bwd_prep_kernel<D, DT>, static_cast<const uint16_t*>(o),
                           static_cast<const uint16_t*>(dout_ptr), lse, p_dq, lse2, dsum);
    if (e != cudaSuccess) return e;
  }
  {
    auto kern = fa_bwd_dq_kernel<D, DT>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::kLaunchSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_dq);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = DqCfg<D>::kLaunchSmem;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, q, k, v, dout, dq_ptr, p_dq);
    if (e != cudaSuccess) return e;
  }
  {
    auto kern = fa_bwd_dkdv_kernel<D, DT>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, KvCfg<D>::kLaunchSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_kv);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = KvCfg<D>::kLaunchSmem;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, q, k, v, dout, dk, dv, p_kv);
  }
  return e;
}

}  // namespace bwd
}  // namespace fa

// Explicit instantiation (PREFIX empty) or its declaration (PREFIX extern).
#define FA_BWD_INSTANTIATE(PREFIX, D, DT)                                                      \
  PREFIX template cudaError_t fa::bwd::launch_fa_bwd<D, DT>(                                   \
      const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, void*,   \
      const CUtensorMap&, const CUtensorMap&, const void*, const void*,                        \
      const float*, float*, float*, const fa::bwd::BwdParams&, const fa::bwd::BwdParams&, int, \
      int, int, cudaStream_t);
