/*
 * fa_kernel.cuh -- FlashAttention forward kernel for sm_103a.
 *
 * One persistent CTA per SM walks a static list of work units.  A unit is
 * (batch*head, pair of 128-row query tiles): the two query tiles share every
 * K/V tile that is streamed in, and their softmax work alternates with each
 * other's matrix products on the tensor cores (the MatMul_n || Softmax_(n-1)
 * overlap that "How the CANN runtime splits FlashAttention" describes in its
 * scheduling layer, and the FA3 ping-pong of "ops-transformer FlashAttention
 * build and tuning", section 1.2).
 *
 * Warp roles (12 warps = 3 warpgroups, 384 threads):
 *   warps 0-3  softmax for query tile 0 (one query row per thread, TMEM lanes)
 *   warps 4-7  softmax for query tile 1
 *   warp  8    TMA producer: Q tiles, then K_j, V_j through an NS-slot ring
 *   warp  9    TMEM owner and tcgen05.mma issuer (the whole warp runs the role;
 *              one elected lane issues the products and commits)
 *   warps 10-11 idle
 * The launch gives every thread 168 registers (three warps share each SM
 * sub-partition's register file); the control warpgroup then hands registers
 * to the softmax warpgroups with setmaxnreg (104 / 200; 120 / 192 at D = 64),
 * so that a softmax thread can hold its whole 128-column score row in
 * registers.
 *
 * Tensor memory (512 columns x 128 lanes, fp32):
 *   [0,128)   S for tile 0   (P for tile 0 overwrites its first columns)
 *   [128,256) S for tile 1
 *   [256,384) O for tile 0   [384,512) O for tile 1
 *
 * Per K/V block j and tile t:
 *   S_t = Q_t K_j^T                     (tcgen05.mma, operands from smem)
 *   softmax warps: mask, running max, conditional O rescale, P = 2^(s*c - m),
 *                  row sum, P -> TMEM as 16-bit (or e4m3 x 256)
 *   O_t += P_t V_j                      (tcgen05.mma, A = P from TMEM)
 * This is the FlashAttention-2 loop order of section 1.2 of the Ascend page
 * (Q block outer, K/V inner) with the online normalisation of its section 6.2
 * written in base 2.  The running max is only moved when the block max
 * exceeds it by more than 2^8 (16-bit P) -- P then stays <= 256, which the
 * 16-bit types and the fp32 accumulators hold exactly as well as <= 1, and
 * O/l is unchanged because O and l share the same stale max.
 *
 * Tail and NaN safety (the Hygon retrospective, defects 2 and 3): TMA never
 * reads outside [0, S) of a tensor -- rows past the end are zero-filled by the
 * tensor map bounds -- and masked columns get P = 0 exactly, so stray NaNs
 * in memory past the valid rows cannot reach the accumulators.
 * 64-bit offsets everywhere a row index meets a stride (defect 1).  Masking
 * uses explicit selects, and the library is built without fast-math
 * (defect 8).  P and O are rounded to nearest-even (defect 9).
 */
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <atomic>
#include <cstdint>

#include "fa_ptx.cuh"
#include "fa_tmem_io.cuh"

namespace fa {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // key/value rows per tile
// Kernel modes: the whole pass over dense [B,H,S,D] tensors, the split-KV
// pass (partials in a workspace), packed variable-length sequences, and
// packed queries against a paged K/V cache.
constexpr int kModeDense = 0, kModeSplit = 1, kModeVarlen = 2, kModePaged = 3;
// Paged K/V with each unit's keys split into n_splits chunks (fp32 partials,
// merged by the combine kernel): the partition-and-reduce of paged decoding.
constexpr int kModePagedSplit = 4;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kCorrWarp0 = 12;  // e4m3: the correction warpgroup (warps 12-15)
constexpr uint32_t kTmemCols = 512;
constexpr int kDtF16 = 0, kDtBF16 = 1, kDtE4M3 = 2;

struct KernelParams {
  int64_t B, H, S_q, S_kv;
  int32_t kv_group;     // query heads per key/value head (1 = multi-head)
  int32_t n_kv_blocks;  // ceil(S_kv / 128)
  int32_t n_pairs;      // ceil(ceil(S_q / 128) / 2)
  int32_t num_units;    // work items: B * H * n_pairs * n_splits
  int32_t group_heads;  // heads per scheduling group (1 = head-major order)
  int32_t layout;       // 0 BNSD, 1 BSND
  int32_t causal;
  float scale_log2;     // |scale| * log2(e)
  int32_t neg_scale;    // scale < 0: S is computed as -Q K^T
  uint32_t idesc_qk;    // the S product's instruction descriptor (set by the launcher)
  const float* descale_q;
  const float* descale_k;
  const float* descale_v;
  void* o;
  float* lse;
  uint32_t* err;
  uint64_t wait_limit_ns;
  int32_t n_splits;     // K/V splits per unit (1: no split; outputs go to o / lse)
  float* lse_part;      // split > 1: fp32 [n_splits, B, H, S_q] partial log-sum-exp
  float* o_part;        // paged split: fp32 [n_splits, H, S_q, D] partial O (row stores)
  // Varlen / paged modes (B = 1; S_q = total_q rows of q / o, lse is [H, total_q]).
  const int32_t* cu_q;         // [n_seqs + 1] query row offsets of each sequence
  const int32_t* cu_k;         // [n_seqs + 1] key row offsets (varlen)
  const int32_t* seqused_k;    // [n_seqs] keys of each sequence (paged)
  const int32_t* block_table;  // [n_seqs, max_pages] page of each key block (paged)
  int32_t n_seqs, max_pages, page_size;
  int32_t q_pack_log2;         // GQA packing: a query tile holds 2^q_pack_log2 heads of
                               // each of 128 >> q_pack_log2 tokens (row = token * 2^.. + head)
  int32_t causal_br;           // causal mask aligned bottom-right (key j visible to
                               // query i iff j <= i + S_kv - S_q)
  const int32_t* seq_order;    // paged: sequence of each rank (longest first), or null
  // Dense mode: units u >= solo_base are single query tiles whose key blocks
  // are split over both tile slots (see Item); the pair units they come from
  // are solo_base + (u - solo_base) / 2.
  int32_t solo_base;
};

template <int D, int DT>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr bool kFp8 = (DT == kDtE4M3);
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;
  static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte swizzle chunks");
  static constexpr int kChunks = kRowBytes / 128;    // 128-byte column chunks per row
  static constexpr int kBoxElems = 128 / kElem;       // elements in one TMA box row
  static constexpr int kChunkBytes = 128 * 128;       // one box: 128 rows x 128 bytes
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kUK = kFp8 ? 32 : 16;          // K of one UMMA instruction
  static constexpr int kQKSteps = D / kUK;
  static constexpr int kPVSteps = kBN / kUK;
  static constexpr int kSlots = (kTileBytes >= 32768) ? 4 : 8;
  static constexpr int kQBytes = 2 * kTileBytes;
  // Epilogue staging: per warp one 32-row x 128-byte box of O (64 columns),
  // written by the warp and drained by a TMA store: 8 warps x 4 KB.
  static constexpr int kEpiBoxBytes = 32 * 128;
  static constexpr int kEpiOffset = kQBytes + kSlots * kTileBytes;
  // e4m3: each block's O-rescale factors (per tile, one fp32 per row), handed
  // from the softmax warps to the correction warpgroup.
  static constexpr int kAlphaOffset = kEpiOffset + 8 * kEpiBoxBytes;
  static constexpr int kBarOffset = kAlphaOffset + (kFp8 ? 2 * 128 * 4 : 0);
  static constexpr int kNumBars = 2 * kSlots + 17;
  static constexpr int kSmemBytes = kBarOffset + kNumBars * 8 + 16 + 1024;  // + align slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kFmt = kFp8 ? 0u : (DT == kDtBF16 ? 1u : 0u);
  static constexpr uint32_t kIdescQK = umma_idesc(kFmt, false, kBM, kBN);
  // The same product with B = K negated (instruction descriptor bit 14):
  // S = -Q K^T, for a negative scale (the softmax then works with |scale|,
  // so that its row maximum of the scores is that of the scaled ones).
  static constexpr uint32_t kIdescQKNeg = kIdescQK | (1u << 14);
  static constexpr uint32_t kIdescPV = umma_idesc(kFmt, true, kBM, D);
  static constexpr float kRescaleThreshold = kFp8 ? 0.0f : 8.0f;
  // Registers per thread after setmaxnreg: softmax warpgroups / control
  // warpgroup; 256 * softmax + 128 * control = 384 * 168 (the launch budget).
  // ~200 hold a softmax thread's 128-score row; the control roles (item
  // decoding, ring bookkeeping, the issuing warp's barrier probes) need ~100.
  // D = 64 runs ~2 % faster with 192 / 120 (2x16x4097x64 causal 86.4 -> 84.8
  // us); D = 128 keeps 200 / 104 (192 / 120 made e4m3 1.8 % slower).
  // e4m3 runs a fourth warpgroup (512 threads, launched at 128 registers;
  // 176 softmax, 72 control, 88 correction -- 184 / 72 / 72 with one O load
  // in flight per round trip was 1.5 % slower):
  // the correction warps, which rescale O when a block moves a row's max --
  // on most e4m3 blocks, since the max moves on every increase (see
  // kRescaleThreshold) -- so that the softmax warps do not wait for O's TMEM
  // round trip (a probe that skipped it: 338 -> 274 us on 1x32x8192 causal).
  // 16-bit P moves the max rarely and keeps three warpgroups.
  static constexpr bool kCorr = kFp8;
  static constexpr int kThreads = kCorr ? 512 : 384;
  static constexpr uint32_t kRegSoftmax = kCorr ? 176 : (D == 64 ? 192 : 200);
  static constexpr uint32_t kRegControl = kCorr ? 72 : (D == 64 ? 120 : 104);
  static constexpr uint32_t kRegCorr = 88;
  static_assert(kCorr ? 2 * kRegSoftmax + kRegControl + kRegCorr == 4 * 128
                      : 256 * kRegSoftmax + 128 * kRegControl == 384 * 168,
                "register budget");
  // log2 of P's scale: e4m3 P holds 256 * p (= 2^(x + 8)), so that weights
  // down to 2^-17 of the row max stay representable; the row sum l then
  // carries the same factor, which O / l cancels and the LSE subtracts.
  static constexpr float kPLog2Scale = kFp8 ? 8.0f : 0.0f;
  static constexpr uint32_t kTmemS = 0, kTmemO = 256;
};

// ---------------------------------------------------------------------------
// Static schedule.  Units are grouped by `group_heads` heads; inside a group
// the longest query-tile pairs come first when causal (LPT order) and heads
// vary fastest, so CTAs running at the same time share K/V in L2.  CTA `bid`
// takes unit w*grid + bid in even rounds and w*grid + grid-1-bid in odd
// rounds (a snake that evens out the causal lengths).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int unit_of_round(int w, int grid, int bid) {
  return w * grid + ((w & 1) ? (grid - 1 - bid) : bid);
}

__device__ __forceinline__ void decode_unit(const KernelParams& p, int u, int& bh, int& pair) {
  const int per_group = p.group_heads * p.n_pairs;
  const int g = u / per_group;
  const int r = u - g * per_group;
  const int BH = static_cast<int>(p.B * p.H);
  const int heads = min(p.group_heads, BH - g * p.group_heads);
  const int rank = r / heads;
  bh = g * p.group_heads + (r - rank * heads);
  pair = p.causal ? (p.n_pairs - 1 - rank) : rank;
}

// K/V blocks query tile `q_tile` needs (0 if the tile has no valid row).
__device__ __forceinline__ int tile_kv_blocks(const KernelParams& p, int q_tile) {
  const int64_t row0 = static_cast<int64_t>(q_tile) * kBM;
  if (row0 >= p.S_q) return 0;
  if (!p.causal) return p.n_kv_blocks;
  const int64_t last_row = min(row0 + (kBM - 1), p.S_q - 1);
  const int64_t max_col = min(last_row, p.S_kv - 1);
  return static_cast<int>(max_col / kBN) + 1;
}

// A CTA's work units in order: unit u of [0, num_units) goes to one CTA by
// the static snake (unit_of_round).  In the varlen / paged modes the snake
// runs over the units that hold query rows only: a query-tile pair past a
// sequence's length is empty, and as a slot of its own it would leave its
// CTA a unit short of the others (32 heads of 32 sequences of 512-8192
// tokens, causal: the busiest CTA 13 % above an even share, 2 % with the
// empty units left out of the count).  Each role walks the list itself; all
// get the same sequence.
template <int kMode>
struct UnitWalk {
  int w = 0;       // this CTA's next round
  int rank = 0;    // varlen / paged: the group (rank, si) the walk is at,
  int si = 0;      // and the units with rows before it
  int64_t k = 0;
  __device__ __forceinline__ bool next(const KernelParams& p, int grid, int bid, int& u) {
    // (A single pair index -- decoding, short prompts -- leaves only
    // sequences without queries empty: the plain snake, without the walk's
    // loads on every unit's path (they cost 2 % on decoding).)
    if (kMode < kModeVarlen || p.n_pairs <= 1) {
      u = unit_of_round(w, grid, bid);
      ++w;
      return u < p.num_units;
    } else {
      // Units with rows, counted in list order, that this CTA takes next.
      const int64_t t = static_cast<int64_t>(w) * grid + ((w & 1) ? (grid - 1 - bid) : bid);
      const int groups = static_cast<int>(p.H) >> p.q_pack_log2;
      const int ns = kMode == kModePagedSplit ? p.n_splits : 1;
      const int64_t gsz = static_cast<int64_t>(groups) * ns;  // units per (rank, sequence)
      const int tile_log2 = 7 - p.q_pack_log2;                  // tokens per query tile
      while (rank < p.n_pairs) {
        const int pair = p.n_pairs - 1 - rank;
        const int seq = p.seq_order ? min(max(p.seq_order[si], 0), p.n_seqs - 1) : si;
        const int64_t q_len =
            min(max(static_cast<int64_t>(p.cu_q[seq + 1]) - p.cu_q[seq], int64_t(0)), p.S_q);
        const int64_t tiles = (q_len + (int64_t(1) << tile_log2) - 1) >> tile_log2;
        if (pair < (tiles + 1) / 2) {
          if (t < k + gsz) {
            // The same unit index decode_item takes: ((rank * n_seqs + si)
            // * groups + head group) * n_splits + split.
            u = static_cast<int>((static_cast<int64_t>(rank) * p.n_seqs + si) * gsz + (t - k));
            ++w;
            return true;
          }
          k += gsz;
        }
        if (++si == p.n_seqs) {
          si = 0;
          ++rank;
        }
      }
      return false;
    }
  }
};

// Work item u = (unit, split): the unit's K/V blocks are cut into n_splits
// chunks of equal length; the item covers blocks [lo, lo + chunk) and tile t
// processes n[t] of them (0: nothing for that tile).  With n_splits = 1 an
// item is a unit and lo = 0.
struct Item {
  int bh, pair, split, lo;
  int n[2];
  // A solo item (dense mode, the last round of a schedule that would leave
  // SMs idle) is one query tile, qt, whose key blocks are split over both
  // tile slots: slot t takes blocks [b[t], b[t] + n[t]); the epilogue merges
  // the two halves.  Otherwise b[0] = b[1] = lo.
  bool solo;
  int qt;
  int b[2];
  // Varlen / paged modes: the unit's sequence, its query / key lengths, the
  // packed row of its first query / key, and the causal offset (0 top-left,
  // S_kv - S_q bottom-right).
  int seq;
  int64_t q_len, k_len, q_row0, k_row0, off;
};

// K/V blocks that query tile q_tile of a sequence needs (varlen / paged); the
// tile covers tokens [q_tile * T, q_tile * T + T), T = 128 >> q_pack_log2.
__device__ __forceinline__ int var_tile_kv_blocks(const KernelParams& p, const Item& it, int q_tile) {
  const int64_t tok_per_tile = kBM >> p.q_pack_log2;
  const int64_t row0 = static_cast<int64_t>(q_tile) * tok_per_tile;
  if (row0 >= it.q_len || it.k_len <= 0) return 0;
  if (!p.causal) return static_cast<int>((it.k_len + kBN - 1) / kBN);
  const int64_t last_row = min(row0 + (tok_per_tile - 1), it.q_len - 1);
  const int64_t max_col = min(last_row + it.off, it.k_len - 1);
  return max_col < 0 ? 0 : static_cast<int>(max_col / kBN) + 1;
}

template <int kMode>
__device__ __forceinline__ Item decode_item(const KernelParams& p, int u) {
  static_assert(kMode >= kModeDense && kMode <= kModePagedSplit, "kernel mode");
  constexpr bool kSplit = kMode == kModeSplit;
  Item it;
  if constexpr (kMode >= kModeVarlen) {
    constexpr bool kVarSplit = kMode == kModePagedSplit;
    const int split = kVarSplit ? u % p.n_splits : 0;
    u = kVarSplit ? u / p.n_splits : u;
    // unit = (query-tile pair, sequence, head group), pairs outermost and
    // the last pairs first: only long sequences have high pairs, and when
    // causal a sequence's last pairs see the most keys, so the costliest
    // units start early (longest-first order).  Within a pair the sequences
    // follow seq_order when given (longest keys first).  Pairs past a
    // sequence's length are empty.  A head group is 2^q_pack_log2 query heads (those of
    // one key/value head when packed, else one head); bh is its index.
    const int groups = static_cast<int>(p.H) >> p.q_pack_log2;
    const int per_rank = p.n_seqs * groups;
    const int rank = u / per_rank;
    const int rem = u - rank * per_rank;
    const int si = rem / groups;  // the sequence's place in the order
    it.seq = p.seq_order ? min(max(p.seq_order[si], 0), p.n_seqs - 1) : si;
    it.bh = rem - si * groups;
    it.pair = p.n_pairs - 1 - rank;
    it.split = 0;
    it.lo = 0;
    // Lengths are clamped to what the tensors can hold, so that offsets
    // that make no sense cost no more than a full pass and never move a
    // store outside the outputs (stores also check rows against [0, S_q)).
    const int64_t q0 = p.cu_q[it.seq], q1 = p.cu_q[it.seq + 1];
    it.q_row0 = q0;
    it.q_len = min(max(q1 - q0, int64_t(0)), p.S_q);
    if constexpr (kMode == kModeVarlen) {
      const int64_t k0 = p.cu_k[it.seq], k1 = p.cu_k[it.seq + 1];
      it.k_row0 = k0;
      it.k_len = min(max(k1 - k0, int64_t(0)), p.S_kv);
    } else {
      it.k_row0 = 0;
      it.k_len = min(max(static_cast<int64_t>(p.seqused_k[it.seq]), int64_t(0)),
                     static_cast<int64_t>(p.max_pages) * p.page_size);
    }
    it.off = p.causal_br ? it.k_len - it.q_len : 0;
    it.n[0] = var_tile_kv_blocks(p, it, 2 * it.pair);
    it.n[1] = var_tile_kv_blocks(p, it, 2 * it.pair + 1);
    it.solo = false;
    it.qt = 2 * it.pair;
    if constexpr (kVarSplit) {
      // This item: key blocks [lo, lo + chunk) of the unit; a split past the
      // sequence's blocks is empty (its partials get zero weight).
      const int nmax = max(it.n[0], it.n[1]);
      const int chunk = (nmax + p.n_splits - 1) / p.n_splits;
      it.split = split;
      it.lo = split * chunk;
      const int hi = min(nmax, it.lo + chunk);
      it.n[0] = max(0, min(it.n[0], hi) - it.lo);
      it.n[1] = max(0, min(it.n[1], hi) - it.lo);
    }
    it.b[0] = it.b[1] = it.lo;
    return it;
  }
  it.seq = 0;
  it.q_len = p.S_q;
  it.k_len = p.S_kv;
  it.q_row0 = 0;
  it.k_row0 = 0;
  it.off = 0;
  int unit = kSplit ? u / p.n_splits : u;
  it.split = kSplit ? u - unit * p.n_splits : 0;
  it.solo = false;
  int solo_tile = 0;
  if constexpr (kMode == kModeDense) {
    if (u >= p.solo_base) {
      unit = p.solo_base + ((u - p.solo_base) >> 1);
      solo_tile = (u - p.solo_base) & 1;
      it.solo = true;
    }
  }
  decode_unit(p, unit, it.bh, it.pair);
  const int f0 = tile_kv_blocks(p, 2 * it.pair), f1 = tile_kv_blocks(p, 2 * it.pair + 1);
  if (it.solo) {
    const int f = solo_tile ? f1 : f0;  // 0: a tile with no row
    it.qt = 2 * it.pair + solo_tile;
    it.lo = 0;
    it.n[0] = (f + 1) >> 1;
    it.n[1] = f - it.n[0];
    it.b[0] = 0;
    it.b[1] = it.n[0];
    return it;
  }
  const int nmax = max(f0, f1);
  const int chunk = kSplit ? (nmax + p.n_splits - 1) / p.n_splits : nmax;
  it.lo = it.split * chunk;
  const int hi = min(nmax, it.lo + chunk);
  it.n[0] = max(0, min(f0, hi) - it.lo);
  it.n[1] = max(0, min(f1, hi) - it.lo);
  it.qt = 2 * it.pair;
  it.b[0] = it.b[1] = it.lo;
  return it;
}

// TMA coordinates of (column c0, row s) of head (b, h): BNSD maps are
// {D, S, H, B}, BSND maps are {D, H, S, B}.
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                         int layout, int32_t c0, int32_t s, int32_t h, int32_t b) {
  if (layout == 0)
    tma_load_4d(dst, map, bar, c0, s, h, b);
  else
    tma_load_4d(dst, map, bar, c0, h, s, b);
}
// A query tile: read once, so marked evict-first in L2.
__device__ __forceinline__ void tma_q_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                           int layout, int32_t c0, int32_t s, int32_t h, int32_t b,
                                           uint64_t pol) {
  if (layout == 0)
    tma_load_4d_hint(dst, map, bar, c0, s, h, b, pol);
  else
    tma_load_4d_hint(dst, map, bar, c0, h, s, b, pol);
}

struct Bars {
  uint32_t base;
  int ns;
  __device__ uint32_t full(int s) const { return base + 8u * s; }
  __device__ uint32_t empty(int s) const { return base + 8u * (ns + s); }
  __device__ uint32_t q_full() const { return base + 8u * (2 * ns); }
  __device__ uint32_t q_empty() const { return base + 8u * (2 * ns + 1); }
  __device__ uint32_t s_full(int t) const { return base + 8u * (2 * ns + 2 + t); }
  __device__ uint32_t p_half(int t, int h) const { return base + 8u * (2 * ns + 4 + 2 * t + h); }
  __device__ uint32_t o_done(int t) const { return base + 8u * (2 * ns + 8 + t); }
  __device__ uint32_t drain() const { return base + 8u * (2 * ns + 10); }
  // Solo items: slot 1's row state is in shared memory / slot 0 has read
  // slot 1's O (one arrival per thread of the warpgroup).
  __device__ uint32_t solo_ml() const { return base + 8u * (2 * ns + 11); }
  __device__ uint32_t solo_read() const { return base + 8u * (2 * ns + 12); }
  // e4m3 correction: tile t's rescale factors of the block are in shared
  // memory / its O is rescaled (one per block and tile).
  __device__ uint32_t alpha_ready(int t) const { return base + 8u * (2 * ns + 13 + t); }
  __device__ uint32_t o_ready(int t) const { return base + 8u * (2 * ns + 15 + t); }
};

// Short bounded wait used only while tearing down after an abort: it ignores
// the abort flag and reports nothing.
__device__ __forceinline__ void mbar_wait_teardown(uint32_t bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit) return;
  }
}

// ---------------------------------------------------------------------------
// Producer (one warp; one elected lane issues): Q pair, then K_0, V_0, K_1,
// V_1, ... into the ring.
// ---------------------------------------------------------------------------
// Paged K/V: the 128 keys of block j of sequence `seq` come from one page
// (page_size >= 128) or from 128 / page_size pages, one TMA box each.  Page
// indices past the sequence's last page are clamped to it (their keys are
// masked); the block table is read only within the sequence's pages.  The
// producer looks a block's pages up once for its K and V tiles, one block
// ahead of their loads, in 32-bit arithmetic (keys < 2^31): the lookups of a
// single thread would otherwise hold up the ring.
struct PagedBlock {
  int32_t page[8];   // the pages of the block's sub-blocks (128 / rows of them)
  int32_t in_page;   // first key of the block inside its page (page_size >= 128)
};

__device__ __forceinline__ void paged_lookup(const KernelParams& p, const int32_t* table,
                                             uint32_t last_page, int j, PagedBlock& pb) {
  const uint32_t ps = static_cast<uint32_t>(p.page_size);
  const uint32_t key0 = static_cast<uint32_t>(j) * kBN;
  const uint32_t pidx0 = key0 / ps;
  pb.in_page = ps >= kBN ? static_cast<int32_t>(key0 - pidx0 * ps) : 0;
  const int nsub = ps >= kBN ? 1 : static_cast<int>(kBN / ps);  // 1, 2, 4 or 8
#pragma unroll
  for (int sub = 0; sub < 8; ++sub)
    if (sub < nsub) pb.page[sub] = table[min(pidx0 + sub, last_page)];
}

template <int D, int DT>
__device__ __forceinline__ void paged_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                           const KernelParams& p, const PagedBlock& pb,
                                           int32_t hk) {
  using C = Cfg<D, DT>;
  const int rows = p.page_size < kBN ? p.page_size : kBN;
  const int nsub = kBN / rows;
#pragma unroll
  for (int sub = 0; sub < 8; ++sub) {
    if (sub >= nsub) break;
    for (int c = 0; c < C::kChunks; ++c)
      tma_load_4d(dst + c * C::kChunkBytes + sub * rows * 128, map, bar, c * C::kBoxElems, hk,
                  pb.in_page, pb.page[sub]);
  }
}

template <int D, int DT, int kMode>
__device__ void producer_role(const KernelParams& p, const CUtensorMap* tmQ,
                              const CUtensorMap* tmK, const CUtensorMap* tmV, uint32_t sQ,
                              uint32_t sRing, const Bars& bars, const WaitCtl& wc) {
  using C = Cfg<D, DT>;
  // The whole warp runs this role; one elected lane arms the barriers and
  // issues the copies (see elect_one).
  const bool leader = elect_one();
  uint32_t ring = 0, it = 0;
  bool ok = true;
  const uint64_t pol_stream = l2_policy_evict_first();
  const int grid = gridDim.x, bid = blockIdx.x;
  UnitWalk<kMode> walk;
  for (int u; ok && walk.next(p, grid, bid, u);) {
    const Item item = decode_item<kMode>(p, u);
    const int bh = item.bh, pair = item.pair;
    // First query head of the tile (varlen / paged: of the head group) and
    // its key/value head; the Q tile's first row.
    const int32_t b = kMode >= kModeVarlen ? 0 : static_cast<int32_t>(bh / p.H);
    const int32_t h = kMode >= kModeVarlen ? (bh << p.q_pack_log2) : static_cast<int32_t>(bh % p.H);
    const int32_t hk = h / p.kv_group;  // key/value head of query head h
    const int32_t tok_per_tile = kMode >= kModeVarlen ? (kBM >> p.q_pack_log2) : kBM;
    const int n0 = item.n[0], n1 = item.n[1];
    const int nmax = max(n0, n1);
    if (nmax == 0) continue;            // an empty split: no MMA work
    if (!mbar_wait(bars.q_empty(), (it & 1u) ^ 1u, wc)) { ok = false; break; }
    if constexpr (kMode == kModeDense) {
      if (item.solo) {
        // One Q tile (into slot 0's buffer), then K of each slot's first
        // block, then per step: V of each slot's block, K of each slot's next.
        if (leader) mbar_arrive_expect_tx(bars.q_full(), C::kTileBytes);
        if (leader)
          for (int c = 0; c < C::kChunks; ++c)
            tma_q_tile(sQ + c * C::kChunkBytes, tmQ, bars.q_full(), p.layout, c * C::kBoxElems,
                       item.qt * kBM, h, b, pol_stream);
        ++it;
        auto load = [&](int kv, int blk) -> bool {
          const int slot = static_cast<int>(ring % C::kSlots);
          if (!mbar_wait(bars.empty(slot), ((ring / C::kSlots) & 1u) ^ 1u, wc)) return false;
          if (leader) mbar_arrive_expect_tx(bars.full(slot), C::kTileBytes);
          if (leader)
            for (int c = 0; c < C::kChunks; ++c)
              tma_tile(sRing + slot * C::kTileBytes + c * C::kChunkBytes, kv == 0 ? tmK : tmV,
                       bars.full(slot), p.layout, c * C::kBoxElems, blk * kBN, hk, b);
          ++ring;
          return true;
        };
        ok = load(0, item.b[0]) && (n1 == 0 || load(0, item.b[1]));
        for (int j = 0; j < n0 && ok; ++j) {
          ok = load(1, item.b[0] + j) && (j >= n1 || load(1, item.b[1] + j));
          if (ok && j + 1 < n0) ok = load(0, item.b[0] + j + 1) && (j + 1 >= n1 || load(0, item.b[1] + j + 1));
        }
        continue;
      }
    }
    if (leader)
      mbar_arrive_expect_tx(bars.q_full(),
                            (n0 > 0 ? C::kTileBytes : 0) + (n1 > 0 ? C::kTileBytes : 0));
    for (int t = 0; t < 2 && leader; ++t) {
      if ((t == 0 ? n0 : n1) == 0) continue;
      for (int c = 0; c < C::kChunks; ++c)
        tma_q_tile(sQ + t * C::kTileBytes + c * C::kChunkBytes, tmQ, bars.q_full(), p.layout,
                   c * C::kBoxElems, static_cast<int32_t>(item.q_row0) + (2 * pair + t) * tok_per_tile,
                   h, b, pol_stream);
    }
    ++it;
    // Paged: the sequence's block-table row and last page; block j + 1's
    // pages are looked up while block j's tiles are in flight.
    constexpr bool kPagedMode = kMode == kModePaged || kMode == kModePagedSplit;
    const int32_t* table = kPagedMode ? p.block_table + static_cast<int64_t>(item.seq) * p.max_pages
                                      : nullptr;
    uint32_t last_page = 0;
    PagedBlock pb;
    if constexpr (kPagedMode) {
      const uint32_t n_pages = static_cast<uint32_t>(
          max((item.k_len + p.page_size - 1) / p.page_size, int64_t(1)));
      last_page = min(n_pages, static_cast<uint32_t>(p.max_pages)) - 1u;
      paged_lookup(p, table, last_page, item.lo, pb);
    }
    for (int j = 0; j < nmax && ok; ++j) {
      for (int kv = 0; kv < 2; ++kv) {
        const int slot = static_cast<int>(ring % C::kSlots);
        if (!mbar_wait(bars.empty(slot), ((ring / C::kSlots) & 1u) ^ 1u, wc)) { ok = false; break; }
        if (leader) mbar_arrive_expect_tx(bars.full(slot), C::kTileBytes);
        const CUtensorMap* map = kv == 0 ? tmK : tmV;
        if constexpr (kPagedMode) {
          if (leader)
            paged_tile<D, DT>(sRing + slot * C::kTileBytes, map, bars.full(slot), p, pb, hk);
          if (kv == 1 && j + 1 < nmax) paged_lookup(p, table, last_page, item.lo + j + 1, pb);
        } else if (leader) {
          for (int c = 0; c < C::kChunks; ++c)
            tma_tile(sRing + slot * C::kTileBytes + c * C::kChunkBytes, map, bars.full(slot),
                     p.layout, c * C::kBoxElems,
                     static_cast<int32_t>(item.k_row0) + (item.lo + j) * kBN, hk, b);
        }
        ++ring;
      }
    }
  }
  if (!ok) {
    // Let loads already in flight land before the CTA's shared memory goes away.
    const uint32_t first = ring > static_cast<uint32_t>(C::kSlots) ? ring - C::kSlots : 0u;
    for (uint32_t r = first; r < ring; ++r)
      mbar_wait_teardown(bars.full(r % C::kSlots), (r / C::kSlots) & 1u, 20000000ull);
    if (it > 0) mbar_wait_teardown(bars.q_full(), (it - 1) & 1u, 20000000ull);
  }
}

// ---------------------------------------------------------------------------
// MMA issuer (one warp; one elected lane issues).
// ---------------------------------------------------------------------------
// S_t = Q_t K^T: K = D in kQKSteps instructions, 32 bytes of K each (inside
// a 128-byte swizzle chunk, then the next 16 KB chunk).  qlo / klo are the low
// descriptor words of the Q tile and the K slot.
template <int D, int DT>
__device__ __forceinline__ void issue_qk(bool leader, uint32_t d_tmem, uint32_t qlo, uint32_t klo,
                                         uint32_t idesc) {
  using C = Cfg<D, DT>;
  constexpr uint32_t hi = umma_desc_hi_sw128(1024);
#pragma unroll
  for (int kk = 0; kk < C::kQKSteps; ++kk) {
    constexpr int kStepBytes = 32;
    const uint32_t off = static_cast<uint32_t>(((kk * kStepBytes / 128) * C::kChunkBytes +
                                                (kk * kStepBytes) % 128) >> 4);
    if (leader)
      umma_ss_w<C::kFp8>(d_tmem, qlo + off, hi, klo + off, hi, idesc, kk > 0 ? 1u : 0u);
  }
}

// O_t (+)= P_t V for keys [64h, 64h+64) (half h of the block): A = P_t from
// TMEM (kUK elements of K = 8 columns per step), B = V rows [kk*kUK, +kUK),
// MN-major (128-byte rows; LBO = next column chunk).
template <int D, int DT, int H>
__device__ __forceinline__ void issue_pv_half(bool leader, uint32_t o_tmem, uint32_t p_tmem,
                                              uint32_t vlo, uint32_t accumulate) {
  using C = Cfg<D, DT>;
  constexpr uint32_t hi = umma_desc_hi_sw128(1024);
  constexpr int kHalf = C::kPVSteps / 2;
#pragma unroll
  for (int kk = H * kHalf; kk < (H + 1) * kHalf; ++kk) {
    const uint32_t off = static_cast<uint32_t>((kk * C::kUK * 128) >> 4);
    if (leader)
      umma_ts_w<C::kFp8>(o_tmem, p_tmem + kk * 8, vlo + off, hi, C::kIdescPV,
                         kk > 0 ? 1u : accumulate);
  }
}

// e4m3: whether tile slot t's keys are one block that takes the softmax's
// masked path (the same test as the softmax's) -- the first tile under a
// causal mask, keys shorter than a block: rows there may see only a few
// keys, and P's residual is added for them.
template <int kMode>
__device__ __forceinline__ bool refine_tile(const KernelParams& p, const Item& it, int t) {
  const int n = t ? it.n[1] : it.n[0];
  if (n != 1) return false;
  const int q_tile = it.solo ? it.qt : 2 * it.pair + t;
  const int shift = kMode >= kModeVarlen ? p.q_pack_log2 : 0;
  const int64_t tile_row0 = static_cast<int64_t>(q_tile) * (kBM >> shift);
  const int64_t col0 = static_cast<int64_t>((t ? it.b[1] : it.b[0]) + n - 1) * kBN;
  return (col0 + kBN > it.k_len) || (p.causal && col0 + (kBN - 1) > tile_row0 + it.off);
}

// e4m3: O_t += P_lo V, P_lo = the residual of P's rounding that the softmax
// writes in the 32 columns after P for a tile refine_tile selects.
template <int D, int DT>
__device__ __forceinline__ void issue_pv_residual(bool leader, uint32_t o_tmem, uint32_t p_tmem,
                                                  uint32_t vlo) {
  using C = Cfg<D, DT>;
  if constexpr (C::kFp8) {
    constexpr uint32_t hi = umma_desc_hi_sw128(1024);
#pragma unroll
    for (int kk = 0; kk < C::kPVSteps; ++kk) {
      const uint32_t off = static_cast<uint32_t>((kk * C::kUK * 128) >> 4);
      if (leader) umma_ts_w<true>(o_tmem, p_tmem + 32 + kk * 8, vlo + off, hi, C::kIdescPV, 1u);
    }
  }
}

// Ring position: slot index and the parity of its current use.
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  template <int NS>
  __device__ __forceinline__ void advance() {
    if (++slot == NS) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// The products of a solo item (see Item): both tile slots multiply the one
// Q tile (slot 0's buffer), slot t over its own key blocks, in the ring
// order the producer loads them.  Returns false if a wait gave up.
template <int D, int DT>
__device__ bool mma_solo_unit(bool leader, const Item& item, RingPos& rp, uint32_t (&p_phase)[2],
                              uint32_t (&o_rphase)[2],
                              uint32_t q_lo, uint32_t k_lo0, uint32_t v_lo0, const uint32_t (&tS)[2],
                              const uint32_t (&tO)[2], const bool (&rf)[2], uint32_t idesc_qk,
                              const Bars& bars, const WaitCtl& wc) {
  using C = Cfg<D, DT>;
  constexpr uint32_t kTileW = C::kTileBytes >> 4;
  const int n[2] = {item.n[0], item.n[1]};  // n[0] >= n[1], n[0] >= 1
  RingPos k[2], v[2];
  k[0] = rp;
  rp.advance<C::kSlots>();
  k[1] = k[0];
  if (n[1] > 0) {
    k[1] = rp;
    rp.advance<C::kSlots>();
  }
  if (!mbar_wait(bars.full(k[0].slot), k[0].phase, wc)) return false;
  if (n[1] > 0 && !mbar_wait(bars.full(k[1].slot), k[1].phase, wc)) return false;
  tc_fence_after();
  issue_qk<D, DT>(leader, tS[0], q_lo, k_lo0 + k[0].slot * kTileW, idesc_qk);
  umma_commit_if(leader, bars.s_full(0));
  if (n[1] > 0) {
    issue_qk<D, DT>(leader, tS[1], q_lo, k_lo0 + k[1].slot * kTileW, idesc_qk);
    umma_commit_if(leader, bars.s_full(1));
    umma_commit_if(leader, bars.empty(k[1].slot));
  }
  umma_commit_if(leader, bars.empty(k[0].slot));
  if (n[0] == 1) umma_commit_if(leader, bars.q_empty());
  for (int j = 0; j < n[0]; ++j) {
    v[0] = rp;
    rp.advance<C::kSlots>();
    if (j < n[1]) {
      v[1] = rp;
      rp.advance<C::kSlots>();
    }
    if (j + 1 < n[0]) {
      k[0] = rp;
      rp.advance<C::kSlots>();
    }
    if (j + 1 < n[1]) {
      k[1] = rp;
      rp.advance<C::kSlots>();
    }
    for (int t = 0; t < 2; ++t) {
      if (j >= n[t]) continue;
      const RingPos& vt = t ? v[1] : v[0];
      const RingPos& kt = t ? k[1] : k[0];
      if (!mbar_wait(bars.p_half(t, 0), p_phase[t], wc)) return false;
      if constexpr (C::kCorr) {
        if (!mbar_wait(bars.o_ready(t), o_rphase[t], wc)) return false;
        o_rphase[t] ^= 1u;
      }
      if (!mbar_wait(bars.full(vt.slot), vt.phase, wc)) return false;
      tc_fence_after();
      issue_pv_half<D, DT, 0>(leader, tO[t], tS[t], v_lo0 + vt.slot * kTileW, j > 0 ? 1u : 0u);
      if (!mbar_wait(bars.p_half(t, 1), p_phase[t], wc)) return false;
      tc_fence_after();
      p_phase[t] ^= 1u;
      issue_pv_half<D, DT, 1>(leader, tO[t], tS[t], v_lo0 + vt.slot * kTileW, 1u);
      if (j + 1 < n[t]) {
        if (!mbar_wait(bars.full(kt.slot), kt.phase, wc)) return false;
        tc_fence_after();
        issue_qk<D, DT>(leader, tS[t], q_lo, k_lo0 + kt.slot * kTileW, idesc_qk);
        umma_commit_if(leader, bars.s_full(t));
      } else {
        if (t ? rf[1] : rf[0])
          issue_pv_residual<D, DT>(leader, tO[t], tS[t], v_lo0 + vt.slot * kTileW);
        umma_commit_if(leader, bars.o_done(t));
      }
    }
    umma_commit_if(leader, bars.empty(v[0].slot));
    if (j < n[1]) umma_commit_if(leader, bars.empty(v[1].slot));
    if (j + 1 < n[0]) umma_commit_if(leader, bars.empty(k[0].slot));
    if (j + 1 < n[1]) umma_commit_if(leader, bars.empty(k[1].slot));
    if (j + 2 == n[0]) umma_commit_if(leader, bars.q_empty());
  }
  return true;
}

template <int D, int DT, int kMode>
__device__ void mma_role(const KernelParams& p, uint32_t tmem, uint32_t sQ, uint32_t sRing,
                         const Bars& bars, const WaitCtl& wc) {
  using C = Cfg<D, DT>;
  // The whole warp runs this role (its control flow is warp-uniform: every
  // lane sees the same barrier states); one elected lane issues the products
  // and commits.
  const bool leader = elect_one();
  constexpr uint32_t kTileW = C::kTileBytes >> 4;  // one tile, in descriptor units
  const uint32_t q_lo[2] = {umma_desc_lo(sQ, 16), umma_desc_lo(sQ, 16) + kTileW};
  const uint32_t k_lo0 = umma_desc_lo(sRing, 16);               // K-major view of slot 0
  const uint32_t v_lo0 = umma_desc_lo(sRing, C::kChunkBytes);   // MN-major view of slot 0
  const uint32_t tS[2] = {tmem + C::kTmemS, tmem + C::kTmemS + kBN};
  const uint32_t tO[2] = {tmem + C::kTmemO, tmem + C::kTmemO + 128};
  // The S product's descriptor, chosen by the launcher: -Q K^T for a
  // negative scale.  (Read from the parameters: selecting it here, or
  // instantiating this role per sign, measured 1-2 % slower on e4m3.)
  const uint32_t idesc_qk = p.idesc_qk;
  RingPos rp;
  uint32_t it = 0;
  uint32_t p_phase[2] = {0u, 0u};
  uint32_t o_rphase[2] = {0u, 0u};  // e4m3: o_ready phases
  bool ok = true;
  const int grid = gridDim.x, bid = blockIdx.x;
  UnitWalk<kMode> walk;
  for (int u; ok && walk.next(p, grid, bid, u);) {
    const Item item = decode_item<kMode>(p, u);
    const int n[2] = {item.n[0], item.n[1]};
    const int nmax = max(n[0], n[1]);
    if (nmax == 0) continue;
    if (!mbar_wait(bars.q_full(), it & 1u, wc)) { ok = false; break; }
    ++it;
    // e4m3: tiles whose last block adds P's rounding residual.
    const bool rf0 = C::kFp8 && refine_tile<kMode>(p, item, 0);
    const bool rf1 = C::kFp8 && refine_tile<kMode>(p, item, 1);
    if constexpr (kMode == kModeDense) {
      if (item.solo) {
        const bool rf[2] = {rf0, rf1};
        if (!mma_solo_unit<D, DT>(leader, item, rp, p_phase, o_rphase, q_lo[0], k_lo0, v_lo0, tS, tO, rf,
                                  idesc_qk, bars, wc)) {
          ok = false;
          break;
        }
        continue;
      }
    }
    // Prologue: S_t = Q_t K_0^T for both tiles.
    int slotK = rp.slot;
    if (!mbar_wait(bars.full(slotK), rp.phase, wc)) { ok = false; break; }
    rp.advance<C::kSlots>();
    tc_fence_after();
    for (int t = 0; t < 2; ++t) {
      if (n[t] == 0) continue;
      issue_qk<D, DT>(leader, tS[t], q_lo[t], k_lo0 + slotK * kTileW, idesc_qk);
      umma_commit_if(leader, bars.s_full(t));
    }
    umma_commit_if(leader, bars.empty(slotK));
    if (nmax == 1) umma_commit_if(leader, bars.q_empty());
    for (int j = 0; j < nmax; ++j) {
      const int slotV = rp.slot;
      const uint32_t phV = rp.phase;
      rp.advance<C::kSlots>();
      const bool has_next = j + 1 < nmax;
      int slotKn = slotK;
      uint32_t phK = 0;
      if (has_next) {
        slotKn = rp.slot;
        phK = rp.phase;
        rp.advance<C::kSlots>();
      }
      bool v_ready = false, k_ready = !has_next;
      // This warp's issue sets the pace, and a blocking wait costs it about as
      // much as a product even when the barrier has long completed (the
      // loads run blocks ahead, and the softmax is usually done).  So every
      // barrier the block needs is first probed with non-blocking tests
      // issued together, whose latencies overlap; a blocking wait runs only
      // for one that has not completed yet.  (Skipping the K and V waits
      // altogether -- unsafe, measured once as a bound -- took the 4 x 32 x
      // 4096 x 128 bf16 pass from 697 to 647 us.)  P comes in two halves: the
      // first half's product runs while the softmax computes the second.
      // bit 0 / 1: first half of P of tile 0 / 1, bit 2: V_j, bit 3: K_{j+1}.
      // (e4m3: the softmax sets the pace and the blocking waits are kept.)
      uint32_t done = 0u;
      if constexpr (!C::kFp8) {
        done = (mbar_test_wait(bars.p_half(0, 0), p_phase[0]) ? 1u : 0u) |
               (mbar_test_wait(bars.p_half(1, 0), p_phase[1]) ? 2u : 0u) |
               (mbar_test_wait(bars.full(slotV), phV) ? 4u : 0u) |
               (mbar_test_wait(bars.full(slotKn), phK) ? 8u : 0u);
      }
      for (int t = 0; t < 2; ++t) {
        if (j >= n[t]) continue;
        if (!((done >> t) & 1u) && !mbar_wait(bars.p_half(t, 0), p_phase[t], wc)) {
          ok = false;
          break;
        }
        // e4m3: the correction warps have rescaled O_t for this block.
        if constexpr (C::kCorr) {
          if (!mbar_wait(bars.o_ready(t), o_rphase[t], wc)) { ok = false; break; }
          o_rphase[t] ^= 1u;
        }
        if (!v_ready) {
          if (!(done & 4u) && !mbar_wait(bars.full(slotV), phV, wc)) { ok = false; break; }
          v_ready = true;
        }
        tc_fence_after();
        issue_pv_half<D, DT, 0>(leader, tO[t], tS[t], v_lo0 + slotV * kTileW, j > 0 ? 1u : 0u);
        if (!mbar_wait(bars.p_half(t, 1), p_phase[t], wc)) { ok = false; break; }
        tc_fence_after();
        p_phase[t] ^= 1u;
        issue_pv_half<D, DT, 1>(leader, tO[t], tS[t], v_lo0 + slotV * kTileW, 1u);
        if (j + 1 < n[t]) {
          if (!k_ready) {
            if (!(done & 8u) && !mbar_wait(bars.full(slotKn), phK, wc)) { ok = false; break; }
            k_ready = true;
            tc_fence_after();
          }
          issue_qk<D, DT>(leader, tS[t], q_lo[t], k_lo0 + slotKn * kTileW, idesc_qk);
          umma_commit_if(leader, bars.s_full(t));
        } else {
          if (t ? rf1 : rf0) issue_pv_residual<D, DT>(leader, tO[t], tS[t], v_lo0 + slotV * kTileW);
          umma_commit_if(leader, bars.o_done(t));
        }
      }
      if (!ok) break;
      // V_j's and K_{j+1}'s slots go back to the producer once every product
      // that reads them has completed.  16-bit: when tile 1 issued S_1(j+1)
      // above, the commit that signals it covers all of them, and tile 1's
      // softmax warps, which wait for that signal anyway, hand the slots back
      // (two commits fewer for this warp); otherwise, and always for e4m3
      // (whose softmax sets the pace: 346 against 332 us on 1 x 32 x 8192
      // causal when it releases), this warp commits them.
      const bool released_by_softmax = !C::kFp8 && j + 1 < n[1];
      if (!released_by_softmax) umma_commit_if(leader, bars.empty(slotV));
      if (has_next) {
        // Every tile that uses K_{j+1} has issued its S by now (a tile with
        // n_t = j + 1 never does), but K_{j+1} may still be unread if no tile
        // needed it: wait for it before handing its slot back.
        if (!k_ready && !(done & 8u) && !mbar_wait(bars.full(slotKn), phK, wc)) { ok = false; break; }
        if (!released_by_softmax) umma_commit_if(leader, bars.empty(slotKn));
        if (j + 2 == nmax) umma_commit_if(leader, bars.q_empty());
      }
      slotK = slotKn;
    }
  }
  // Drain: every MMA issued above completes before TMEM is released.
  umma_commit_if(leader, bars.drain());
  mbar_wait_teardown(bars.drain(), 0u, ok ? 2000000000ull : 20000000ull);
}

// ---------------------------------------------------------------------------
// Softmax / correction / epilogue (warps 0-7; one query row per thread).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void st_shared_f1(uint32_t addr, float a) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(a) : "memory");
}
__device__ __forceinline__ float ld_shared_f1(uint32_t addr) {
  float a;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(a) : "r"(addr) : "memory");
  return a;
}

__device__ __forceinline__ void st_shared_f2(uint32_t addr, float a, float b) {
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ void ld_shared_f2(uint32_t addr, float& a, float& b) {
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(a), "=f"(b) : "r"(addr) : "memory");
}

// One K/V block of the softmax for one query row (the thread's TMEM lane):
// row max, running-max update with conditional O rescale, P = 2^(s*sl2 - m)
// in two halves, each signalled once written, row sum.  Instantiated twice --
// with and without the tail/causal mask -- so the unmasked copy, which almost
// every block runs, is one contiguous straight-line body.
template <int D, int DT, bool kMasked>
__device__ __forceinline__ void softmax_block(float (&s)[128], int lim, int j, float sl2,
                                              float& m_run, float& l, uint32_t tS, uint32_t tO,
                                              uint32_t alpha_slot, const Bars& bars, int t) {
  using C = Cfg<D, DT>;
  // Masked columns become -inf: they drop out of the max and give p = 0.
  if constexpr (kMasked) {
#pragma unroll
    for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : -CUDART_INF_F;
  }
  // 3-input max tree over the 128 scores (depth 5, ~64 instructions).
  float t43[43];
#pragma unroll
  for (int i = 0; i < 42; ++i) t43[i] = max3(s[3 * i], s[3 * i + 1], s[3 * i + 2]);
  t43[42] = fmaxf(s[126], s[127]);
  float t15[15];
#pragma unroll
  for (int i = 0; i < 14; ++i) t15[i] = max3(t43[3 * i], t43[3 * i + 1], t43[3 * i + 2]);
  t15[14] = t43[42];
  const float t5a = max3(t15[0], t15[1], t15[2]), t5b = max3(t15[3], t15[4], t15[5]);
  const float t5c = max3(t15[6], t15[7], t15[8]), t5d = max3(t15[9], t15[10], t15[11]);
  const float t5e = max3(t15[12], t15[13], t15[14]);
  const float mxb = max3(max3(t5a, t5b, t5c), t5d, t5e);
  const float m_blk = (mxb == -CUDART_INF_F) ? -CUDART_INF_F : mxb * sl2;
  const float m_new = fmaxf(m_run, m_blk);
  // Decide the running max for this block.  On the first block O holds
  // nothing yet (its first PV overwrites it); later the max only moves
  // when it grew past the threshold, and then O and l are rescaled.
  float alpha = 1.0f;
  bool resc = false;
  if (j == 0) {
    m_run = m_new;
  } else if (m_new > m_run + C::kRescaleThreshold) {
    resc = true;
    alpha = ex2(m_run - m_new);
    l *= alpha;
    m_run = m_new;
  }
  const float m_sub = (m_run == -CUDART_INF_F) ? 0.0f : m_run;
  // O_t *= alpha for the rows whose max moved, before any PV of this block
  // accumulates into O (O is complete: the commit that signalled S_j
  // covered the previous PV; this block's PV waits for P below).  e4m3: the
  // correction warps do it (correction_role) while this warp computes P; it
  // hands them the row's factor, 1 when the max did not move.
  if constexpr (C::kCorr) {
    st_shared_f1(alpha_slot, alpha);
    mbar_arrive(bars.alpha_ready(t));
  } else if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t ov[32];
      tmem_ld_x32(tO + 32 * c, ov);
      tmem_wait_ld();
      reg_dep_x32(ov);
#pragma unroll
      for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
      tmem_st_x32(tO + 32 * c, ov);
    }
    tmem_wait_st();
  }
  // p = 2^(s * sl2 - m), in two halves of 64 columns.  After each half its
  // P (16-bit, or e4m3 x 256) goes to TMEM; for e4m3 each half is signalled
  // on its own, so the PV product of the first 64 keys runs while the second
  // half is computed.
  // The loops are straight-line code (no branch inside) so the scheduler
  // can hide MUFU latency across columns.
  const float negm = C::kFp8 ? C::kPLog2Scale - m_sub : -m_sub;
  const uint64_t sl2x2 = f2_pack(sl2, sl2), negm2 = f2_pack(negm, negm);
  uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    // Masked columns already hold -inf (set before the max), and sl2 > 0,
    // so they come out as exactly 0; one loop serves every block.
#pragma unroll
    for (int i = 32 * h; i < 32 * h + 32; ++i) {
      float x0, x1;
      f2_unpack(f2_fma(f2_pack(s[2 * i], s[2 * i + 1]), sl2x2, negm2), x0, x1);
      x0 = ex2(x0);
      x1 = ex2(x1);
      s[2 * i] = x0;
      s[2 * i + 1] = x1;
      if (i & 1) acc1 = f2_add(acc1, f2_pack(x0, x1)); else acc0 = f2_add(acc0, f2_pack(x0, x1));
    }
    if constexpr (C::kFp8) {
      // Masked blocks also write the residual P - e4m3(P), in e4m3, to the
      // next 32 columns; for a tile whose keys are that one block (see
      // refine_tile) the PV product adds it: P then reaches O to 2^-8 instead
      // of 2^-4 -- for rows that see only a few keys, whose weights are not
      // averaged.  (Computing it in every masked block keeps the flag out of
      // the loop: a runtime flag there cost registers.)
      if constexpr (kMasked) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {  // in groups of 8 columns (fewer live registers)
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = 64 * h + 32 * g + 4 * i;
            hi[i] = pack_e4m3x4(s[c], s[c + 1], s[c + 2], s[c + 3]);
            float q0, q1, q2, q3;
            e4m3x4_unpack(hi[i], q0, q1, q2, q3);
            lo[i] = pack_e4m3x4(s[c] - q0, s[c + 1] - q1, s[c + 2] - q2, s[c + 3] - q3);
          }
          tmem_st_x8(tS + 16 * h + 8 * g, hi);
          tmem_st_x8(tS + 32 + 16 * h + 8 * g, lo);
        }
      } else {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = 64 * h + 4 * i;
          pk[i] = pack_e4m3x4(s[c], s[c + 1], s[c + 2], s[c + 3]);
        }
        tmem_st_x16(tS + 16 * h, pk);
      }
    } else {
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int c = 64 * h + 2 * i;
        pk[i] = (DT == kDtF16) ? pack_f16x2(s[c], s[c + 1]) : pack_bf16x2(s[c], s[c + 1]);
      }
      tmem_st_x32(tS + 32 * h, pk);
    }
    // Each half is signalled once written: its product runs while the next
    // half is computed.
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bars.p_half(t, h));
  }
  {
    float x0, x1;
    f2_unpack(f2_add(acc0, acc1), x0, x1);
    l += x0 + x1;
  }}

// Where a row's lse goes: the final lse [B, H, S_q], or -- for a split --
// that split's slice of the fp32 partial lse [n_splits, B, H, S_q].
template <bool kSplit>
__device__ __forceinline__ float* lse_row_base(const KernelParams& p, int split, int bh) {
  if (!kSplit) return p.lse + static_cast<int64_t>(bh) * p.S_q;
  return p.lse_part + (static_cast<int64_t>(split) * p.B * p.H + bh) * p.S_q;
}

__device__ __forceinline__ void st_global_v4(void* ptr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

template <int D, int DT, int kMode>
__device__ void softmax_role(const KernelParams& p, const CUtensorMap* tmO, const CUtensorMap* tmOp,
                             uint32_t tmem, uint32_t sEpi, int warp, int lane, const Bars& bars,
                             const WaitCtl& wc) {
  using C = Cfg<D, DT>;
  const int t = warp >> 2;            // query tile of this warpgroup
  const int wq = warp & 3;            // TMEM lane quarter
  const int r = wq * 32 + lane;       // row inside the tile
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tmem + lane_off + C::kTmemS + t * kBN;
  const uint32_t tO = tmem + lane_off + C::kTmemO + t * 128;
  // e4m3: this row's slot for the block's O-rescale factor.
  const uint32_t alpha_slot =
      sEpi + static_cast<uint32_t>(C::kAlphaOffset - C::kEpiOffset + (t * 128 + r) * 4);
  constexpr bool kVarSplit = kMode == kModePagedSplit;
  constexpr bool kSplit = kMode == kModeSplit;    // dense split: [n*B, H, S_q, D] partials
  constexpr bool split = kSplit || kVarSplit;     // fp32 partial O and lse
  constexpr bool kVar = kMode >= kModeVarlen;
  // The lane that issues this warp's output stores and waits for them (a
  // bulk async-group belongs to the thread that committed it, so the same
  // elected lane does both; see elect_one).
  const bool leader = elect_one();

  float sl2 = p.scale_log2;
  float o_mul = 1.0f;
  if constexpr (C::kFp8) {
    const float dq = p.descale_q ? *p.descale_q : 1.0f;
    const float dk = p.descale_k ? *p.descale_k : 1.0f;
    const float dv = p.descale_v ? *p.descale_v : 1.0f;
    sl2 *= dq * dk;
    o_mul = dv;  // (P's factor 256 is in l too: O / l cancels it)
  }
  // A masked score is -inf and must give p = 0: keep the base-2 scale
  // strictly positive (a zero scale or descale becomes 1e-30, which changes
  // no unmasked exponent by more than ~1e-29 relative).
  sl2 = fmaxf(sl2, 1e-30f);

  uint32_t s_phase = 0u, o_phase = 0u, solo_phase = 0u;
  uint32_t ring_pos = 0u;   // K/V ring positions consumed by earlier items
  const int grid = gridDim.x, bid = blockIdx.x;
  UnitWalk<kMode> walk;
  for (int u; walk.next(p, grid, bid, u);) {
    const Item item = decode_item<kMode>(p, u);
    const int bh = item.bh;
    // A solo item's two slots work on the same tile, qt.
    const int q_tile = item.solo ? item.qt : 2 * item.pair + t;
    const int n = t ? item.n[1] : item.n[0];
    const int blk0 = t ? item.b[1] : item.b[0];  // this slot's first key block
    // Ring position of this item's first K tile; the item's tiles occupy the
    // next 2 * max(n0, n1) positions (K_0, V_0, K_1, V_1, ...), a solo item's
    // 2 * (n0 + n1).
    const uint32_t ring_base = ring_pos;
    ring_pos += item.solo ? 2u * static_cast<uint32_t>(item.n[0] + item.n[1])
                          : 2u * static_cast<uint32_t>(max(item.n[0], item.n[1]));
    // 16-bit: tile 1 hands back the ring slots of V_{j-1} and K_j once S_1(j)
    // is ready (see mma_role): one thread of the warpgroup.
    const bool releaser = !C::kFp8 && t == 1 && !item.solo && threadIdx.x == 128;
    // Tile rows are tokens (dense, split: 128 of one head); varlen / paged
    // with GQA packing: 2^shift heads of each of 128 >> shift tokens.
    const int shift = kVar ? p.q_pack_log2 : 0;
    const int64_t tile_row0 = static_cast<int64_t>(q_tile) * (kBM >> shift);  // first token
    const int64_t row = tile_row0 + (r >> shift);                              // this row's token
    const int hrow = kVar ? (bh << shift) + (r & ((1 << shift) - 1)) : bh;     // and its head
    const int64_t q_len = item.q_len, k_len = item.k_len;
    if (n == 0) {
      // No key of this split is visible to this tile: an empty partial,
      // which the merge gives zero weight.
      if (kSplit && row < p.S_q) lse_row_base<kSplit>(p, item.split, bh)[row] = -CUDART_INF_F;
      if (kVarSplit && row < q_len && item.q_row0 + row < p.S_q && item.q_row0 + row >= 0)
        p.lse_part[(static_cast<int64_t>(item.split) * p.H + hrow) * p.S_q + item.q_row0 + row] =
            -CUDART_INF_F;
      // A varlen / paged tile whose rows see no key at all: O = 0, lse = -inf.
      if (kVar && !kVarSplit && row < q_len && item.q_row0 + row < p.S_q &&
          item.q_row0 + row >= 0) {
        const int64_t grow = item.q_row0 + row;
        uint8_t* orow = static_cast<uint8_t*>(p.o) + ((grow * p.H + hrow) * D) * 2;
        for (int c = 0; c < D / 8; ++c) st_global_v4(orow + 16 * c, 0u, 0u, 0u, 0u);
        p.lse[static_cast<int64_t>(hrow) * p.S_q + grow] = -CUDART_INF_F;
      }
      continue;
    }
    // Key j of the sequence is visible to this row iff j < col_end.
    const int64_t col_end =
        p.causal ? max(min(row + item.off + 1, k_len), int64_t(0)) : k_len;

    float m_run = -CUDART_INF_F, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait(bars.s_full(t), s_phase, wc)) { ok = false; break; }
      s_phase ^= 1u;
      if (releaser && j > 0) {
        mbar_arrive(bars.empty((ring_base + 2u * j - 1u) % C::kSlots));
        mbar_arrive(bars.empty((ring_base + 2u * j) % C::kSlots));
      }
      tc_fence_after();
      // The block's 128 scores: one 128-column load for 16-bit (~1.8 % faster
      // than four of 32 columns); four for e4m3 (2.7 % slower with one).
      float s[128];
      if constexpr (C::kFp8) {
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_x32(tS + 32 * c, sr[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_dep_x32(sr[c]);
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
      } else {
        uint32_t sr[128];
        tmem_ld_x128(tS, sr);
        tmem_wait_ld();
        reg_dep_x128(sr);
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
      }

      const int64_t col0 = static_cast<int64_t>(blk0 + j) * kBN;
      // Block-uniform: does any column of this block need a mask?
      const bool masked = (col0 + kBN > k_len) || (p.causal && col0 + (kBN - 1) > tile_row0 + item.off);
      const int lim = static_cast<int>(max(min(col_end - col0, static_cast<int64_t>(kBN)), int64_t(0)));
      if (masked)
        softmax_block<D, DT, true>(s, lim, j, sl2, m_run, l, tS, tO, alpha_slot, bars, t);
      else
        softmax_block<D, DT, false>(s, kBN, j, sl2, m_run, l, tS, tO, alpha_slot, bars, t);
    }
    if (!ok) break;

    // Epilogue.  O / l goes through a per-warp staging box in shared memory
    // (32 rows x 128 bytes, 128-byte swizzle) and a TMA store whose tensor
    // map clips rows >= S_q: 64 columns of 16-bit output per box, or -- for a
    // split -- 32 columns of the fp32 partial O per box.  Then lse.
    if (!mbar_wait(bars.o_done(t), o_phase, wc)) break;
    o_phase ^= 1u;
    tc_fence_after();
    // Solo item with both slots busy: slot 1 hands its row state (m, l) to
    // slot 0 through its own staging box and waits until slot 0 has read its
    // O from TMEM; slot 0 merges the halves, O = (a0 O0 + a1 O1) / (a0 l0 +
    // a1 l1) with a_i = 2^(m_i - max(m0, m1)), and writes the tile.
    const bool merge = item.solo && item.n[1] > 0;
    float a0 = 1.0f, a1 = 0.0f;
    if (merge) {
      const uint32_t ml = sEpi + static_cast<uint32_t>(4 + wq) * C::kEpiBoxBytes + lane * 8;
      const uint32_t ph = solo_phase;
      solo_phase ^= 1u;
      if (t == 1) {
        if (leader) bulk_wait_group_read0();  // this box's last store has read it
        __syncwarp();
        st_shared_f2(ml, m_run, l);
        tc_fence_before();
        mbar_arrive(bars.solo_ml());
        if (!mbar_wait(bars.solo_read(), ph, wc)) break;
        tc_fence_after();
        continue;
      }
      if (!mbar_wait(bars.solo_ml(), ph, wc)) break;
      tc_fence_after();
      float m1, l1;
      ld_shared_f2(ml, m1, l1);
      const float mm = fmaxf(m_run, m1);
      a0 = (m_run == -CUDART_INF_F) ? 0.0f : ex2(m_run - mm);
      a1 = (m1 == -CUDART_INF_F) ? 0.0f : ex2(m1 - mm);
      l = a0 * l + a1 * l1;
      m_run = mm;
    }
    // (A varlen / paged row that saw no key has l = 0: O = 0.)
    const float inv = (kVar && l == 0.0f) ? 0.0f : o_mul / l;
    const float c0 = a0 * inv, c1 = a1 * inv;  // O = c0 O0 (+ c1 O1 when merging)
    const uint32_t tO1 = tO + 128;               // slot 1's O (read when merging)
    // This warp's 32 rows: tokens [box_row0, box_row0 + box_toks).
    const int box_toks = 32 >> shift;
    const int32_t box_row0 = static_cast<int32_t>(tile_row0) + wq * box_toks;
    const uint32_t stage = sEpi + static_cast<uint32_t>(warp) * C::kEpiBoxBytes;
    const int n_boxes = split ? D / 32 : D / 64;
    const int32_t b = static_cast<int32_t>(bh / p.H), h = static_cast<int32_t>(bh % p.H);
#pragma unroll 1
    for (int bx = 0; bx < n_boxes; ++bx) {
      uint32_t pk[32];
      if (split) {
        uint32_t o0[32];
        tmem_ld_x32(tO + 32 * bx, o0);
        tmem_wait_ld();
        reg_dep_x32(o0);
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = __float_as_uint(__uint_as_float(o0[i]) * inv);
      } else if (merge) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t o0[32], o1[32];
          tmem_ld_x32(tO + 64 * bx + 32 * hf, o0);
          tmem_ld_x32(tO1 + 64 * bx + 32 * hf, o1);
          tmem_wait_ld();
          reg_dep_x32(o0);
          reg_dep_x32(o1);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float x0 = fmaf(__uint_as_float(o1[2 * i]), c1, __uint_as_float(o0[2 * i]) * c0);
            const float x1 = fmaf(__uint_as_float(o1[2 * i + 1]), c1, __uint_as_float(o0[2 * i + 1]) * c0);
            pk[16 * hf + i] = (DT == kDtF16) ? pack_f16x2(x0, x1) : pack_bf16x2(x0, x1);
          }
        }
      } else {
        uint32_t o0[32], o1[32];
        tmem_ld_x32(tO + 64 * bx, o0);
        tmem_ld_x32(tO + 64 * bx + 32, o1);
        tmem_wait_ld();
        reg_dep_x32(o0);
        reg_dep_x32(o1);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a0 = __uint_as_float(o0[2 * i]) * inv, a1 = __uint_as_float(o0[2 * i + 1]) * inv;
          const float c0 = __uint_as_float(o1[2 * i]) * inv, c1 = __uint_as_float(o1[2 * i + 1]) * inv;
          pk[i] = (DT == kDtF16) ? pack_f16x2(a0, a1) : pack_bf16x2(a0, a1);
          pk[16 + i] = (DT == kDtF16) ? pack_f16x2(c0, c1) : pack_bf16x2(c0, c1);
        }
      }
      if constexpr (kVar) {
        // A box that runs past the sequence's last row: per-row stores of
        // the rows inside it (a TMA store would write the next sequence's).
        if (box_row0 + box_toks > q_len) {
          if (row < q_len && item.q_row0 + row < p.S_q && item.q_row0 + row >= 0) {
            uint8_t* orow =
                kVarSplit ? reinterpret_cast<uint8_t*>(
                                p.o_part + ((static_cast<int64_t>(item.split) * p.H + hrow) * p.S_q +
                                            item.q_row0 + row) * D + 32 * bx)
                          : static_cast<uint8_t*>(p.o) +
                                (((item.q_row0 + row) * p.H + hrow) * D + 64 * bx) * 2;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_global_v4(orow + 16 * q, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
          continue;
        }
      }
      // The previous TMA store from this staging box must have read it.
      if (leader) bulk_wait_group_read0();
      __syncwarp();
      // Staging row of this thread's row: the box's element order.  The
      // head-major partial box of a packed tile (heads x tokens) takes row
      // (head, token); every other box is in lane order.
      const int srow = kVarSplit ? ((lane & ((1 << shift) - 1)) * box_toks + (lane >> shift)) : lane;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_shared_v4(stage + srow * 128 + ((q ^ (srow & 7)) << 4), pk[4 * q], pk[4 * q + 1],
                     pk[4 * q + 2], pk[4 * q + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      // Rows past S_q are clipped by the map; a store never starts at a
      // negative row.
      if (leader && (kVar ? (item.q_row0 + box_row0 >= 0 && item.q_row0 + box_row0 < p.S_q)
                             : box_row0 < p.S_q)) {
        if (kVarSplit)
          tma_store_4d(tmOp, stage, 32 * bx, static_cast<int32_t>(item.q_row0) + box_row0,
                       bh << shift, item.split);
        else if (kVar)
          tma_store_4d_hint(tmO, stage, 64 * bx, bh << shift,
                            static_cast<int32_t>(item.q_row0) + box_row0, 0,
                            l2_policy_evict_first());
        else if (split)
          tma_store_4d(tmOp, stage, 32 * bx, box_row0, h, item.split * static_cast<int32_t>(p.B) + b);
        else if (p.layout == 0)  // output tiles are written once: evict-first in L2
          tma_store_4d_hint(tmO, stage, 64 * bx, box_row0, h, b, l2_policy_evict_first());
        else
          tma_store_4d_hint(tmO, stage, 64 * bx, h, box_row0, b, l2_policy_evict_first());
        bulk_commit_group();
      }
    }
    if (merge) {
      // Every read of slot 1's O has completed (each load above was waited).
      tc_fence_before();
      mbar_arrive(bars.solo_read());
    }
    if constexpr (kVar) {
      float* lse_dst = kVarSplit ? p.lse_part + static_cast<int64_t>(item.split) * p.H * p.S_q : p.lse;
      if (row < q_len && item.q_row0 + row < p.S_q && item.q_row0 + row >= 0)
        lse_dst[static_cast<int64_t>(hrow) * p.S_q + item.q_row0 + row] =
            l > 0.0f ? (m_run + log2f(l) - C::kPLog2Scale) * 0.69314718055994531f : -CUDART_INF_F;
    } else if (row < p.S_q) {
      lse_row_base<kSplit>(p, item.split, bh)[row] =
          (m_run + log2f(l) - C::kPLog2Scale) * 0.69314718055994531f;
    }
    tc_fence_before();
  }
  // Every TMA store of this warp has completed before the CTA exits.
  if (leader) bulk_wait_group0();
  __syncwarp();
}

// ---------------------------------------------------------------------------
// e4m3 correction warpgroup (warps 12-15, one TMEM lane quarter each): for
// every block of every tile slot, in the order the issuing warp takes them,
// O_t *= alpha (the row's factor the softmax handed over) when any row of
// the warp's quarter moved its max, then O_t is released for the block's PV
// product.  The softmax warps meanwhile compute P.
// ---------------------------------------------------------------------------
template <int D, int DT, int kMode>
__device__ void correction_role(const KernelParams& p, uint32_t tmem, uint32_t sEpi, int warp,
                                int lane, const Bars& bars, const WaitCtl& wc) {
  using C = Cfg<D, DT>;
  const int wq = warp & 3;
  const int r = wq * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t sAlpha = sEpi + static_cast<uint32_t>(C::kAlphaOffset - C::kEpiOffset);
  uint32_t a_phase[2] = {0u, 0u};
  const int grid = gridDim.x, bid = blockIdx.x;
  UnitWalk<kMode> walk;
  bool ok = true;
  for (int u; ok && walk.next(p, grid, bid, u);) {
    const Item item = decode_item<kMode>(p, u);
    const int nmax = max(item.n[0], item.n[1]);
    for (int j = 0; j < nmax && ok; ++j) {
      for (int t = 0; t < 2; ++t) {
        if (j >= (t ? item.n[1] : item.n[0])) continue;
        if (!mbar_wait(bars.alpha_ready(t), a_phase[t], wc)) { ok = false; break; }
        a_phase[t] ^= 1u;
        const float alpha = ld_shared_f1(sAlpha + static_cast<uint32_t>((t * 128 + r) * 4));
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
          tc_fence_after();
          const uint32_t tO = tmem + lane_off + C::kTmemO + t * 128;
          // Two 32-column loads in flight per round trip (1.5 % faster than
          // one: the issuing warp waits for this before the block's PV).
#pragma unroll 1
          for (int c = 0; c < D / 32; c += 2) {
            uint32_t ov[32], ow[32];
            tmem_ld_x32(tO + 32 * c, ov);
            tmem_ld_x32(tO + 32 * c + 32, ow);
            tmem_wait_ld();
            reg_dep_x32(ov);
            reg_dep_x32(ow);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st_x32(tO + 32 * c, ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ow[i] = __float_as_uint(__uint_as_float(ow[i]) * alpha);
            tmem_st_x32(tO + 32 * c + 32, ow);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.o_ready(t));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int D, int DT, int kMode>
__global__ void __launch_bounds__(Cfg<D, DT>::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const __grid_constant__ CUtensorMap tmOp, const __grid_constant__ KernelParams p) {
  using C = Cfg<D, DT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sRing = base + C::kQBytes;
  const uint32_t sEpi = base + C::kEpiOffset;
  const Bars bars{base + static_cast<uint32_t>(C::kBarOffset), C::kSlots};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBarOffset + C::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    mbar_init(bars.q_full(), 1);
    mbar_init(bars.q_empty(), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bars.s_full(t), 1);
      mbar_init(bars.p_half(t, 0), 128);
      mbar_init(bars.p_half(t, 1), 128);
      mbar_init(bars.o_done(t), 1);
    }
    mbar_init(bars.drain(), 1);
    mbar_init(bars.solo_ml(), 128);
    mbar_init(bars.solo_read(), 128);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bars.alpha_ready(t), 128);
      mbar_init(bars.o_ready(t), 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
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
  // The grid is launched with programmatic stream serialization, so it may
  // start (on SMs the kernel before it leaves idle) while that kernel still
  // runs: nothing below touches global memory before that kernel has
  // completed and its writes are visible.  And the kernel after it -- the
  // next call, or the split merge -- may start its own prologue now, on SMs
  // this grid leaves idle (its own wait guards its memory accesses).  For
  // small problems that hides the launch and prologue of consecutive calls.
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp < kProducerWarp) {
    reg_alloc_inc<C::kRegSoftmax>();
    softmax_role<D, DT, kMode>(p, &tmO, &tmOp, tmem, sEpi, warp, lane, bars, wc);
  } else if (C::kCorr && warp >= kCorrWarp0) {
    reg_alloc_dec<C::kRegCorr>();
    correction_role<D, DT, kMode>(p, tmem, sEpi, warp, lane, bars, wc);
  } else {
    reg_alloc_dec<C::kRegControl>();
    if (warp == kProducerWarp) {
      producer_role<D, DT, kMode>(p, &tmQ, &tmK, &tmV, sQ, sRing, bars, wc);
    } else if (warp == kMmaWarp) {
      mma_role<D, DT, kMode>(p, tmem, sQ, sRing, bars, wc);
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The calling thread's current context (made current if it has none), or
// null (defined with the entry points).
CUcontext current_context(int* dev_out);

// Host-side launcher, one instantiation per (D, dtype, mode).  The kernel's
// shared-memory limit is raised once per device and context, not per call.
template <int D, int DT, int kMode>
cudaError_t launch_fa_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& o, const CUtensorMap& op, const KernelParams& p,
                          int grid, cudaStream_t stream) {
  using C = Cfg<D, DT>;
  auto kern = fa_fwd_kernel<D, DT, kMode>;
  static std::atomic<CUcontext> attr_ctx[64];
  int dev = 0;
  const CUcontext ctx = current_context(&dev);
  if (!ctx || dev < 0 || dev >= 64 || attr_ctx[dev].load(std::memory_order_acquire) != ctx) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (ctx && dev >= 0 && dev < 64) attr_ctx[dev].store(ctx, std::memory_order_release);
  }
  KernelParams pp = p;
  pp.idesc_qk = p.neg_scale ? C::kIdescQKNeg : C::kIdescQK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, o, op, pp);
}

}  // namespace fa

// Explicit instantiation (PREFIX empty) or its declaration (PREFIX extern).
#define FA_FWD_INSTANTIATE(PREFIX, D, DT, MODE)                                              \
  PREFIX template cudaError_t fa::launch_fa_fwd<D, DT, MODE>(                                \
      const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,        \
      const CUtensorMap&, const fa::KernelParams&, int, cudaStream_t);
