// fa_kernel.cuh -- the attention forward kernel for sm_103a.
//
// One persistent CTA per SM walks a list of work items.  An item is a pair
// of 128-row Q tiles of one (batch, head): tile 0 = rows [256p, 256p+128),
// tile 1 = the next 128 rows.  This is the query-block parallelism of the
// FlashAttention v2 work-partitioning diagram (pseudo-code panel, "parallel
// for batch, head, q_block"; core panel item 2: more CTAs along the
// sequence) and its sliced-Q split (each softmax warp owns 32 Q rows and
// half of their S columns; K/V tiles are shared, and the only exchange
// between warps is a row maximum and a row sum between the two halves).
//
// Roles inside the CTA (FlashAttention v4 Blackwell pipeline diagram, the
// producer / MMA / softmax lanes and the pseudo-code panel), 640 threads:
//   warps 0-15  softmax, two groups of eight: warps 0-7 own Q tile 0 and
//               warps 8-15 Q tile 1, so the two tiles' softmax runs
//               concurrently; in a group, warps w and w + 4 split the 128
//               columns of S of the rows of lane quadrant w % 4 (about half
//               the softmax latency of one warp per row); each group also
//               runs its tile's epilogue (O / l, logsumexp)
//   warp  16    MMA issue (one elected lane) + tensor-memory allocation
//   warp  17    TMA producer (one thread): Q tiles and a K/V ring
//   warps 18-19 idle (they complete the fifth warpgroup, whose registers
//               go to the softmax warpgroups through setmaxnreg)
//
// Tensor memory (512 columns x 128 lanes, 32-bit cells):
//   S0 [0,128)   S1 [128,256)   O0 [256,256+D)   O1 [256+D,256+2D)
//   d = 64 only: P0 [384,448)   P1 [448,512)
// S_t = Q_t K_j^T (fp32).  After the softmax reads S_t it writes P_t as
// packed 16-bit pairs -- over the first 64 columns of S_t (d = 128), or in
// P_t's own columns (d = 64) -- and the second MMA takes P_t straight from
// tensor memory: S and P never leave the chip.
//
// MMA issue order per K/V block j (ping-pong between the two Q tiles, so one
// group's softmax overlaps the other group's MMAs), d = 128:
//   S0_{j+1}, PV1_j, S1_{j+1}, PV0_{j+1}
// Each S_t commit also covers the PV_t issued before it, so a softmax group
// that sees S_t(j+1) ready may rescale O_t (PV_t(j) is complete) and the
// MMA does not issue PV_t(j+1) until that group signals P_t ready.
// d = 64 (P apart from S):
//   S0_{j+1}, PV1_{j-1}, S1_{j+1}, PV0_j
// S_t(j+1) is issued as soon as the group has loaded S_t(j) into registers
// (an "S free" barrier), so the group finds it ready when it finishes block
// j; each PV_t commits a "PV done" barrier that the group awaits before it
// writes P_t again or rescales O_t.
//
// Every wait is bounded: after kTimeoutNs without progress the thread sets
// the CTA's abort flag and the device status word, and all roles leave
// their loops; in-flight copies and MMAs are drained before the tensor
// memory is freed, so the context stays usable.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace fa {

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s without progress
constexpr int kMaxSplit = 4;                     // most pieces a split item is cut into
constexpr uint32_t kStatusTimeout = 1u;

struct Params {
  void *o;           // [BH, N, D] 16-bit
  float *lse;        // [BH, N] fp32
  unsigned *status;  // device status word
  int N;             // sequence length
  int BH;            // B * H
  int n_qtiles;      // ceil(N / 128)
  int n_pairs;       // ceil(n_qtiles / 2)
  int n_items;       // BH * n_pairs
  int causal;
  int causal_head_major;  // causal item order: 0 heaviest pair first across heads, 1 head by head
  int causal_tail_heads;  // head by head: the last this many heads go heaviest pair first across them
  float scale_log2;  // scale * log2(e)
  float rescale_thr; // rescale O only when the running max grows by more than this (log2 units)
  // Wave-tail split (non-causal only): the items from
  // split_first on (those of the last, partial round of the persistent
  // grid) are cut into split_k pieces along the key blocks; each piece
  // leaves its O (normalised by its own sum) and row statistics in scratch
  // memory, and the last piece of an item to finish merges them.
  int n_units;          // work units: split_first + (n_items - split_first) * split_k
  int split_first;      // first split item (n_items: none)
  int split_k;          // pieces per split item
  float4 *part_o;       // [piece][D / 4 column groups][256 rows] fp32 x 4
  float *part_st;       // [piece][3][256 rows]: max (log2 units), sum of P, corrected sum
  unsigned *part_cnt;   // [split item]: pieces finished (zero before the launch)
  // rescale counters (kernel variants built with STATS only): [0] (row,
  // block) pairs after a tile's first block whose running max grew past the
  // threshold, [1] all such (row, block) pairs, [2] warp-blocks that ran
  // the O rescale loop, [3] all warp-blocks after a tile's first block
  unsigned long long *stats;
};

// Kernel variants: STAGES = K/V ring slots (0: the default, 4 at d = 128
// and 8 at d = 64), EXPSPLIT = every EXPSPLIT-th pair of the softmax's
// exponentials is evaluated on the FMA pipes (exp2_poly2) instead of the
// special-function unit (0: none), STATS = count rescales (Params::stats).
template <int D, bool BF16, int STAGES = 0, int EXPSPLIT = 0, bool STATS = false>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dim must be 64 or 128");
  static constexpr int kRows = 128;                   // Q rows per tile, keys per block
  static constexpr int kTileBytes = kRows * D * 2;    // one Q, K or V tile
  static constexpr int kHalfBytes = kRows * 64 * 2;   // 64 columns: one 128-byte swizzle span
  static constexpr int kStages = STAGES ? STAGES : ((D == 128) ? 4 : 8);  // K/V ring slots
  static constexpr int kExpSplit = EXPSPLIT;
  static constexpr bool kStats = STATS;
  static_assert(kStages >= 2, "the ring needs two slots");
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 2 * kTileBytes;
  static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
  // barrier indices
  // per Q tile: kQFull + t, kQEmpty + t
  static constexpr int kQFull = 0, kQEmpty = 2, kKVFull = 4, kKVEmpty = 4 + kStages;
  static constexpr int kSFull = 4 + 2 * kStages, kPFull = kSFull + 2, kOFull = kPFull + 2;
  static constexpr int kDrain = kOFull + 2;
  // d = 64: P has tensor-memory columns of its own (there is room), so S_t
  // can be overwritten as soon as the softmax has loaded it.  Two more
  // barriers per tile: S free (kSFree + t, one arrive per warp of the
  // tile's group) and PV done (kPVDone + t, an MMA commit after each PV).
  static constexpr bool kSepP = (D == 64);
  static constexpr int kSFree = kDrain + 1, kPVDone = kSFree + 2;
  static constexpr int kNumBars = kSepP ? kPVDone + 2 : kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag, merge flag
  // softmax row exchange: [tile][parity][half][value][row] floats, 8 KB
  static constexpr int kXchOff = (kMiscOff + 16 + 15) & ~15;
  static constexpr int kSmemBytes = kXchOff + 2 * 2 * 2 * 2 * 128 * 4 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory beyond the per-CTA limit");
  static constexpr uint32_t kTmemCols = 512;
  // tensor-memory column of S_t, O_t and P_t for Q tile t: P_t is packed
  // 16-bit pairs over the first 64 columns of S_t (d = 128), or in its own
  // 64 columns after O (d = 64: S 0-255, O 256-383, P 384-511)
  static __device__ __forceinline__ uint32_t col_s(int t) { return 128u * t; }
  static __device__ __forceinline__ uint32_t col_o(int t) { return 256u + D * t; }
  static __device__ __forceinline__ uint32_t col_p(int t) {
    return kSepP ? 256u + 2u * D + 64u * t : col_s(t);
  }
  static constexpr uint32_t kIdescS = idesc_f16(BF16, false, 128, 128);
  static constexpr uint32_t kIdescO = idesc_f16(BF16, true, 128, D);
  // Five warpgroups -- four of softmax (eight warps per Q tile) and one with
  // the MMA and TMA warps -- launched at 96 registers a thread (five warps
  // share each SMSP's 16384), then setmaxnreg 4 x 128 x 104 + 128 x 56
  // <= 640 x 96.
  static constexpr int kThreads = 640;
  static constexpr int kSoftmaxWarps = 16;
  static constexpr int kMmaWarp = kSoftmaxWarps, kTmaWarp = kSoftmaxWarps + 1;
  static constexpr uint32_t kRegsSoftmax = 104, kRegsOther = 56;
};

struct Item {
  int bh, qt0, n0, n1;
  int j0;     // first K/V block
  int piece;  // -1: a whole item; else the global piece index
};

// Work item -> (head, first Q tile, K/V blocks for each of the two tiles).
// Non-causal items run head-major so CTAs working at the same time share a
// few heads' K/V in L2.  Causal items run heaviest pair first (the pair
// nearest the end of the sequence sees the most keys), across all heads --
// or, where the host found that order no better balanced, head by head
// (heaviest pair first within a head), which keeps each head's K/V in L2
// for all of its pairs; then the last causal_tail_heads heads are taken
// together, heaviest pair first across them, so the light pairs of several
// heads end the launch instead of one head's heavy ones.
__device__ __forceinline__ Item decode_item(int item, const Params &p) {
  Item it;
  int pair;
  if (p.causal && p.causal_head_major) {
    const int g = p.causal_tail_heads;
    const int first = (p.BH - g) * p.n_pairs;
    if (item < first) {
      it.bh = item / p.n_pairs;
      pair = p.n_pairs - 1 - (item - it.bh * p.n_pairs);
    } else {
      const int s = item - first;
      const int level = s / g;
      it.bh = p.BH - g + (s - level * g);
      pair = p.n_pairs - 1 - level;
    }
  } else if (p.causal) {
    const int level = item / p.BH;
    it.bh = item - level * p.BH;
    pair = p.n_pairs - 1 - level;
  } else {
    it.bh = item / p.n_pairs;
    pair = item - it.bh * p.n_pairs;
  }
  it.qt0 = 2 * pair;
  const int qt1 = it.qt0 + 1;
  it.n0 = p.causal ? it.qt0 + 1 : p.n_qtiles;
  it.n1 = (qt1 < p.n_qtiles) ? (p.causal ? qt1 + 1 : p.n_qtiles) : 0;
  return it;
}

// Work unit -> item, with the key-block range of a piece of a split item.
// Piece c of k takes blocks [c * n / k, (c + 1) * n / k) of the n_qtiles.
__device__ __forceinline__ Item decode_unit(int unit, const Params &p) {
  if (unit < p.split_first) {
    Item it = decode_item(unit, p);
    it.j0 = 0;
    it.piece = -1;
    return it;
  }
  const int s = unit - p.split_first;
  const int k = p.split_k;
  const int q = s / k, c = s - q * k;
  Item it = decode_item(p.split_first + q, p);
  const int lo = c * p.n_qtiles / k, hi = (c + 1) * p.n_qtiles / k;
  it.j0 = lo;
  it.n0 = hi - lo;
  it.n1 = it.n1 > 0 ? hi - lo : 0;
  it.piece = s;
  return it;
}

// The work unit a CTA takes in a given round of the persistent loop, or -1.
// Causal rounds alternate direction so the CTA that took the heaviest item
// of one round takes the lightest of the next.
__device__ __forceinline__ int round_item(int round, const Params &p) {
  const int base = round * static_cast<int>(gridDim.x);
  const int off = (p.causal && (round & 1)) ? static_cast<int>(gridDim.x - 1 - blockIdx.x)
                                            : static_cast<int>(blockIdx.x);
  const int idx = base + off;
  return idx < p.n_units ? idx : -1;
}

__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned *status, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        atomicOr(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// Bounded wait for phase `parity` of barrier `bar`; false = give up.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         unsigned *status, uint64_t timeout_ns = kTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, abort_flag, status, timeout_ns);
}

// Drain wait: bounded by time only (the awaited copy or MMA needs nothing
// from other threads to finish).  Giving up is reported like any other
// timeout, so the caller learns that memory may still have been in use.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           unsigned *status) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kTimeoutNs) {
      *abort_flag = 1;
      atomicOr(status, kStatusTimeout);
      return;
    }
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
}

// 2^x for a pair of x on the FMA pipes, for the share of the softmax's
// exponentials taken off the special-function unit (the FlashAttention v4
// Blackwell pipeline diagram, pseudo-code panel and v3 -> v4 comparison:
// exp is emulated in software for part of the elements).  Cody-Waite
// split x = n + f, n = round(x): adding 1.5 * 2^23 rounds x to an integer
// and leaves n in the low mantissa bits of the sum, so those bits shifted
// into the exponent field scale p(f) by 2^n.  p(f) ~ 2^f on [-1/2, 1/2] is
// a minimax fit of the relative error (Remez exchange, computed by
// fit_exp2_poly.py in this directory): degree 3 (7.5e-5) for bf16
// probabilities, degree 4 (2.6e-6) for fp16.  x is clamped at -127 and a
// result whose exponent would go below zero is flushed to +0 by an integer
// max, so masked logits (-inf) give exactly 0 as the hardware ex2 does.
template <bool BF16>
__device__ __forceinline__ void exp2_poly2(uint64_t x2, float &e0, float &e1) {
  constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
  float x0, x1;
  f2_split(x2, x0, x1);
  const uint64_t xc = f2(fmaxf(x0, -127.0f), fmaxf(x1, -127.0f));
  const uint64_t t = fadd2(xc, f2(kRound, kRound));            // round(x) in the low bits
  const uint64_t n = fadd2(t, f2(-kRound, -kRound));           // round(x), exactly
  const uint64_t f = ffma2(n, f2(-1.0f, -1.0f), xc);            // x - n, exactly
  uint64_t q;
  if constexpr (BF16) {
    q = ffma2(f, f2(5.517166853e-02f, 5.517166853e-02f), f2(2.426111251e-01f, 2.426111251e-01f));
    q = ffma2(q, f, f2(6.932609677e-01f, 6.932609677e-01f));
    q = ffma2(q, f, f2(9.999280572e-01f, 9.999280572e-01f));
  } else {
    q = ffma2(f, f2(9.570102207e-03f, 9.570102207e-03f), f2(5.591785908e-02f, 5.591785908e-02f));
    q = ffma2(q, f, f2(2.402474433e-01f, 2.402474433e-01f));
    q = ffma2(q, f, f2(6.931217909e-01f, 6.931217909e-01f));
    q = ffma2(q, f, f2(9.999992847e-01f, 9.999992847e-01f));
  }
  float q0, q1, t0, t1;
  f2_split(q, q0, q1);
  f2_split(t, t0, t1);
  e0 = __int_as_float(max(__float_as_int(q0) + (__float_as_int(t0) << 23), 0));
  e1 = __int_as_float(max(__float_as_int(q1) + (__float_as_int(t1) << 23), 0));
}

// Stores a segment of NC 16-byte chunks (NC = 8: 128 bytes, NC = 4: 64
// bytes) of each of a warp's 32 rows (lane = row) so that every store
// instruction writes whole segments: within each group of NC lanes an NC x NC
// transpose of the chunks (log2(NC) xor-shuffle stages) leaves lane i of the
// group holding chunk i of the group's NC rows.  Row r of the warp is at
// row0 + r * stride bytes; rows r >= rows_valid are not written.
template <int NC>
__device__ __forceinline__ void store_rows(uint4 (&v)[NC], uint8_t *row0, size_t stride,
                                           int rows_valid, uint32_t lane) {
  static_assert(NC == 4 || NC == 8, "4 or 8 chunks per row");
#pragma unroll
  for (int k = NC / 2; k >= 1; k >>= 1) {
    const bool hi = (lane & k) != 0;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      if (c & k) continue;
      const uint4 send = hi ? v[c] : v[c | k];
      uint4 recv;
      recv.x = __shfl_xor_sync(0xffffffffu, send.x, k);
      recv.y = __shfl_xor_sync(0xffffffffu, send.y, k);
      recv.z = __shfl_xor_sync(0xffffffffu, send.z, k);
      recv.w = __shfl_xor_sync(0xffffffffu, send.w, k);
      if (hi) v[c] = recv;
      else v[c | k] = recv;
    }
  }
  const int g = static_cast<int>(lane) / NC, i = static_cast<int>(lane) % NC;
#pragma unroll
  for (int r = 0; r < NC; ++r) {
    const int row = NC * g + r;
    if (row < rows_valid)
      *reinterpret_cast<uint4 *>(row0 + static_cast<size_t>(row) * stride + 16 * i) = v[r];
  }
}

template <int D, bool BF16, int STAGES = 0, int EXPSPLIT = 0, bool STATS = false>
__global__ void __launch_bounds__(Cfg<D, BF16, STAGES, EXPSPLIT, STATS>::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using C = Cfg<D, BF16, STAGES, EXPSPLIT, STATS>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte-swizzled tiles.
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (sbase - raw);

  const uint32_t bars = sbase + C::kBarOff;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_base_slot = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(bar(C::kKVFull + i), 1);
      mbar_init(bar(C::kKVEmpty + i), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kQFull + t), 1);
      mbar_init(bar(C::kQEmpty + t), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kSFull + t), 1);
      mbar_init(bar(C::kPFull + t), 8);  // one arrive per softmax warp of the tile's group
      mbar_init(bar(C::kOFull + t), 1);
    }
    mbar_init(bar(C::kDrain), 1);
    if constexpr (C::kSepP) {
      for (int t = 0; t < 2; ++t) {
        mbar_init(bar(C::kSFree + t), 8);  // one arrive per softmax warp of the tile's group
        mbar_init(bar(C::kPVDone + t), 1);
      }
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::kTmaWarp && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_base_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;
  // launched as a programmatic dependent: nothing above touches global
  // memory; wait here for the previous kernel in the stream to complete
  // (and its writes to be visible), then let the next one be scheduled (its
  // CTAs take SMs only as this grid's CTAs leave them, and wait likewise)
  griddep_wait();
  griddep_launch_dependents();

  if (warp >= C::kSoftmaxWarps) {
    // Each role's code sits under its own setmaxnreg, so the compiler sizes
    // it for that role's register budget only.
    regs_dec<C::kRegsOther>();
    if (warp == C::kTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t slot = 0, phase = 0, q_phase[2] = {0, 0};
      uint32_t kv_loads = 0, q_loads[2] = {0, 0};
      bool ok = true;
      for (int round = 0; ok && round * static_cast<int>(gridDim.x) < p.n_units; ++round) {
        const int item = round_item(round, p);
        if (item < 0) continue;
        const Item it = decode_unit(item, p);
        // Each Q tile's buffer is released by its own last S MMA of the
        // previous item, so tile 0's next tile can load while tile 1 still
        // computes.
        const int nq = it.n1 > 0 ? 2 : 1;
        for (int t = 0; ok && t < nq; ++t) {
          if (!(ok = wait_bar(bar(C::kQEmpty + t), q_phase[t] ^ 1u, abort_flag, p.status))) break;
          q_phase[t] ^= 1u;
          mbar_arrive_expect_tx(bar(C::kQFull + t), C::kTileBytes);
          for (int h = 0; h < D / 64; ++h)
            tma_load_3d(sbase + C::kQOff + t * C::kTileBytes + h * C::kHalfBytes, &tm_q,
                        bar(C::kQFull + t), h * 64, (it.qt0 + t) * 128, it.bh, pol_q);
          ++q_loads[t];
        }
        if (!ok) break;
        const int n_max = it.n0 > it.n1 ? it.n0 : it.n1;
        for (int j = 0; ok && j < n_max; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            if (!(ok = wait_bar(bar(C::kKVEmpty + slot), phase ^ 1u, abort_flag, p.status))) break;
            mbar_arrive_expect_tx(bar(C::kKVFull + slot), C::kTileBytes);
            const CUtensorMap *m = kv ? &tm_v : &tm_k;
            for (int h = 0; h < D / 64; ++h)
              tma_load_3d(sbase + C::kKVOff + slot * C::kTileBytes + h * C::kHalfBytes, m,
                          bar(C::kKVFull + slot), h * 64, (it.j0 + j) * 128, it.bh, pol_kv);
            ++kv_loads;
            if (++slot == C::kStages) {
              slot = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Drain: every issued copy must land before the CTA's shared memory
      // can be released.  Slot s received loads s, s+S, s+2S, ... < kv_loads.
      for (int s = 0; s < C::kStages; ++s) {
        if (static_cast<uint32_t>(s) < kv_loads) {
          const uint32_t cnt = (kv_loads - s + C::kStages - 1) / C::kStages;
          wait_drain(bar(C::kKVFull + s), (cnt - 1) & 1u, abort_flag, p.status);
        }
      }
      for (int t = 0; t < 2; ++t)
        if (q_loads[t]) wait_drain(bar(C::kQFull + t), (q_loads[t] - 1) & 1u, abort_flag, p.status);
    }
    } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------- MMA issue
    // The whole warp runs this loop (waits included) and one elected lane
    // issues the MMAs and commits: a converged warp issues faster than a
    // lone divergent lane.
    {
      const uint32_t leader = elect_one();
      uint32_t slot = 0, phase = 0, q_phase[2] = {0, 0}, p_phase[2] = {0, 0};
      bool ok = true;
      auto advance = [&]() {
        if (++slot == C::kStages) {
          slot = 0;
          phase ^= 1u;
        }
      };
      // Descriptors are built once; per MMA only the K-step offset (in
      // 16-byte units, inside the 14-bit address field) is added.
      const uint64_t kdesc0 = smem_desc_sw128(0, 16, 1024);             // Q, K: K-major
      const uint64_t vdesc0 = smem_desc_sw128(0, C::kHalfBytes, 1024);  // V: MN-major
      auto issue_s = [&](int t, uint32_t kslot) {
        const uint64_t qd = kdesc0 + ((sbase + C::kQOff + t * C::kTileBytes) >> 4);
        const uint64_t kd = kdesc0 + ((sbase + C::kKVOff + kslot * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kHalfBytes + (kk & 3) * 32) >> 4;
          mma_ss_if(leader, tmem + C::col_s(t), qd + off, kd + off, C::kIdescS, kk > 0);
        }
      };
      auto issue_pv = [&](int t, uint32_t vslot, bool acc) {
        const uint64_t vd = vdesc0 + ((sbase + C::kKVOff + vslot * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk) {
          mma_ts_if(leader, tmem + C::col_o(t), tmem + C::col_p(t) + kk * 8, vd + kk * (2048 >> 4),
                 C::kIdescO, (acc || kk > 0) ? 1u : 0u);
        }
      };
      // Two issue loops, kept flat: d = 128 (P over S) here, d = 64 (P in its
      // own columns) in the else branch below.
      if constexpr (!C::kSepP) {
      // The loop is rotated so that the iteration boundary (and the release
      // of a K slot) falls right after PV0's MMAs are queued: between the end
      // of S1's issue and the start of PV0's there is then only one commit
      // and one wait, and the tensor core's short queue does not run dry.
      for (int round = 0; ok && round * static_cast<int>(gridDim.x) < p.n_units; ++round) {
        const int item = round_item(round, p);
        if (item < 0) continue;
        const Item it = decode_unit(item, p);
        const int n_max = it.n0 > it.n1 ? it.n0 : it.n1;
        if (!(ok = wait_bar(bar(C::kQFull + 0), q_phase[0], abort_flag, p.status))) break;
        q_phase[0] ^= 1u;
        // K_0 and V_0 positions in the ring
        uint32_t ks = slot, kph = phase;
        advance();
        uint32_t vs = slot, vph = phase;
        advance();
        if (!(ok = wait_bar(bar(C::kKVFull + ks), kph, abort_flag, p.status))) break;
        tc_fence_after();
        issue_s(0, ks);
        mma_commit_if(leader, bar(C::kSFull + 0));
        if (it.n0 == 1) mma_commit_if(leader, bar(C::kQEmpty + 0));
        if (it.n1 > 0) {
          if (!(ok = wait_bar(bar(C::kQFull + 1), q_phase[1], abort_flag, p.status))) break;
          q_phase[1] ^= 1u;
          tc_fence_after();
          issue_s(1, ks);
          mma_commit_if(leader, bar(C::kSFull + 1));
          if (it.n1 == 1) mma_commit_if(leader, bar(C::kQEmpty + 1));
        }
        mma_commit_if(leader, bar(C::kKVEmpty + ks));
        // PV0(0) (tile 0 always has at least one block)
        if (!(ok = wait_bar(bar(C::kKVFull + vs), vph, abort_flag, p.status))) break;
        if (!(ok = wait_bar(bar(C::kPFull + 0), p_phase[0], abort_flag, p.status))) break;
        p_phase[0] ^= 1u;
        tc_fence_after();
        issue_pv(0, vs, false);
        for (int j = 0; j < n_max; ++j) {
          // queued: PV0(j)
          const bool more = j + 1 < n_max;
          if (more) {
            ks = slot;
            kph = phase;
            advance();
            if (!(ok = wait_bar(bar(C::kKVFull + ks), kph, abort_flag, p.status))) break;
            tc_fence_after();
          }
          // tile 0: S0(j+1), or the end of tile 0 (PV0(n0-1) is already queued)
          if (j + 1 < it.n0) {
            issue_s(0, ks);
            mma_commit_if(leader, bar(C::kSFull + 0));
            if (j + 2 == it.n0) mma_commit_if(leader, bar(C::kQEmpty + 0));  // last S0
          } else if (j + 1 == it.n0) {
            mma_commit_if(leader, bar(C::kOFull + 0));
          }
          // tile 1: PV1(j)
          if (j < it.n1) {
            if (!(ok = wait_bar(bar(C::kPFull + 1), p_phase[1], abort_flag, p.status))) break;
            p_phase[1] ^= 1u;
            tc_fence_after();
            issue_pv(1, vs, j > 0);
          }
          mma_commit_if(leader, bar(C::kKVEmpty + vs));  // V_j read by PV0(j) and PV1(j)
          uint32_t nvs = 0;
          if (more) {  // V_{j+1}: checked now, before S1's MMAs fill the queue
            nvs = slot;
            const uint32_t nvph = phase;
            advance();
            if (!(ok = wait_bar(bar(C::kKVFull + nvs), nvph, abort_flag, p.status))) break;
          }
          // tile 1: S1(j+1), or the end of tile 1
          if (j + 1 < it.n1) {
            issue_s(1, ks);
            mma_commit_if(leader, bar(C::kSFull + 1));
            if (j + 2 == it.n1) mma_commit_if(leader, bar(C::kQEmpty + 1));  // last S1
          } else if (j + 1 == it.n1) {
            mma_commit_if(leader, bar(C::kOFull + 1));
          }
          if (more) {
            // tile 0: PV0(j+1)
            if (j + 1 < it.n0) {
              if (!(ok = wait_bar(bar(C::kPFull + 0), p_phase[0], abort_flag, p.status))) break;
              p_phase[0] ^= 1u;
              tc_fence_after();
              issue_pv(0, nvs, true);
            }
            mma_commit_if(leader, bar(C::kKVEmpty + ks));  // K_{j+1} read by S0(j+1) and S1(j+1)
            vs = nvs;
          }
        }
      }
      } else {  // d = 64
      // d = 64, P in its own columns.  Per block j the MMAs go
      //   S0(j+1), PV1(j-1), S1(j+1), PV0(j)
      // (the order in which their inputs become ready).  S_t(j+1) waits only
      // until the softmax has loaded S_t(j) into registers (S free), so each
      // softmax group finds its next S ready when it finishes a block;
      // PV_t(j) waits for P_t(j) and commits PV done, which the softmax
      // awaits before it writes P_t(j+1) or rescales O_t.  An item's first S
      // waits for the S free of the previous item's last block, so it
      // overlaps that block and its epilogue.
      uint32_t ring = 0;  // K/V ring entries taken by earlier items: K_j at ring + 2j, V_j next
      uint32_t sfree_par[2] = {0, 0};
      bool s_held[2] = {false, false};  // S_t holds an S whose S free is still to be awaited
      auto kv_slot = [&](uint32_t idx) -> uint32_t { return idx % C::kStages; };
      auto wait_kv = [&](uint32_t idx) {
        return wait_bar(bar(C::kKVFull + kv_slot(idx)), (idx / C::kStages) & 1u, abort_flag,
                        p.status);
      };
      // S_t(j) of a tile with n blocks: its commits, and the Q release after the last
      auto s_mma = [&](int t, int j, int n) -> bool {
        if (s_held[t]) {
          if (!wait_bar(bar(C::kSFree + t), sfree_par[t], abort_flag, p.status)) return false;
          sfree_par[t] ^= 1u;
        }
        if (!wait_kv(ring + 2u * j)) return false;
        tc_fence_after();
        issue_s(t, kv_slot(ring + 2u * j));
        mma_commit_if(leader, bar(C::kSFull + t));
        if (j + 1 == n) mma_commit_if(leader, bar(C::kQEmpty + t));
        s_held[t] = true;
        return true;
      };
      auto pv_mma = [&](int t, int j) -> bool {
        if (!wait_bar(bar(C::kPFull + t), p_phase[t], abort_flag, p.status)) return false;
        p_phase[t] ^= 1u;
        if (!wait_kv(ring + 2u * j + 1u)) return false;
        tc_fence_after();
        issue_pv(t, kv_slot(ring + 2u * j + 1u), j > 0);
        mma_commit_if(leader, bar(C::kPVDone + t));
        return true;
      };
      for (int round = 0; ok && round * static_cast<int>(gridDim.x) < p.n_units; ++round) {
        const int item = round_item(round, p);
        if (item < 0) continue;
        const Item it = decode_unit(item, p);
        const int n0 = it.n0, n1 = it.n1;  // n1: 0 (no tile 1), n0 or n0 + 1
        const int n_max = n0 > n1 ? n0 : n1;
        if (!(ok = wait_bar(bar(C::kQFull + 0), q_phase[0], abort_flag, p.status))) break;
        q_phase[0] ^= 1u;
        if (!(ok = s_mma(0, 0, n0))) break;
        if (n1 > 0) {
          if (!(ok = wait_bar(bar(C::kQFull + 1), q_phase[1], abort_flag, p.status))) break;
          q_phase[1] ^= 1u;
          if (!(ok = s_mma(1, 0, n1))) break;
        }
        mma_commit_if(leader, bar(C::kKVEmpty + kv_slot(ring)));  // K_0
        for (int j = 0; j < n_max; ++j) {
          if (j + 1 < n0 && !(ok = s_mma(0, j + 1, n0))) break;
          if (j >= 1 && j - 1 < n1) {
            if (!(ok = pv_mma(1, j - 1))) break;
            mma_commit_if(leader, bar(C::kKVEmpty + kv_slot(ring + 2u * (j - 1) + 1u)));  // V_{j-1}
          }
          if (j + 1 < n1 && !(ok = s_mma(1, j + 1, n1))) break;
          if (j + 1 < n_max) mma_commit_if(leader, bar(C::kKVEmpty + kv_slot(ring + 2u * (j + 1))));  // K_{j+1}
          if (j < n0) {
            if (!(ok = pv_mma(0, j))) break;
            if (j >= n1)  // V_j has no tile-1 reader
              mma_commit_if(leader, bar(C::kKVEmpty + kv_slot(ring + 2u * j + 1u)));
          }
        }
        if (!ok) break;
        if (n1 > 0 && n1 == n_max) {  // PV1 of tile 1's last block
          if (!(ok = pv_mma(1, n1 - 1))) break;
          mma_commit_if(leader, bar(C::kKVEmpty + kv_slot(ring + 2u * (n1 - 1) + 1u)));
        }
        ring += 2u * static_cast<uint32_t>(n_max);
      }
      }
      // Drain: all issued MMAs complete before tensor memory is freed.
      mma_commit_if(leader, bar(C::kDrain));
      wait_drain(bar(C::kDrain), 0, abort_flag, p.status);
    }
    }
  } else {
    regs_inc<C::kRegsSoftmax>();
    // ------------------------------------------ softmax, column split
    // Two groups of eight warps, one per Q tile (warps 0-7: tile 0, 8-15:
    // tile 1), so the two tiles' softmax runs concurrently.  In a group,
    // warp w takes the 32 rows of tensor-memory lane quadrant q = w % 4 (one
    // thread per row) and the 64 columns [64h, 64h + 64) of S,
    // h = (w / 4) % 2: two warps share a quadrant's rows, so the softmax of a
    // block takes about half as long as with one warp per row.  The two
    // warps of a quadrant exchange partial row maxima (and, at the end,
    // partial row sums) through shared memory.
    const int t = warp >> 3;  // this group's Q tile
    const int q = warp & 3, hf = (warp >> 2) & 1;
    const uint32_t lane_base = q * 32u;
    const int row = static_cast<int>(lane_base + lane);
    const uint32_t t_lane = tmem + (lane_base << 16);
    float *xch = reinterpret_cast<float *>(smem + C::kXchOff);  // [tile][parity][half][value][row]
    auto xslot = [&](uint32_t par, int h, int val) {
      return xch + (((t * 2 + par) * 2 + h) * 2 + val) * 128 + row;
    };
    // named barrier of the quadrant's two warps in this group (1..8)
    const uint32_t pair_bar = 1u + static_cast<uint32_t>(q) + 4u * static_cast<uint32_t>(t);
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory"); };
    // all sixteen softmax warps (named barrier 9)
    auto softmax_sync = [&]() { asm volatile("bar.sync 9, 512;" ::: "memory"); };
    volatile unsigned *merge_flag = reinterpret_cast<volatile unsigned *>(smem + C::kMiscOff + 8);
    // Merge of the pieces of a split item, tile t, this thread's row and
    // half of the columns: with M the largest of the pieces' maxima, piece
    // c weighs r_c 2^(m_c - M) (its corrected sum) in O, and the logsumexp
    // is M + log2(sum_c l_c 2^(m_c - M)) (in log2 units).  Reads go to L2
    // (other SMs wrote the pieces).
    auto merge = [&](const Item &it, int t) {
      const int k = p.split_k;
      const int first = (it.piece / k) * k;
      const int prow_in_item = t * 128 + row;
      float m_c[kMaxSplit], w[kMaxSplit];
      float M = -INFINITY;
#pragma unroll
      for (int c = 0; c < kMaxSplit; ++c) {
        m_c[c] = -INFINITY;
        if (c < k) {
          m_c[c] = __ldcg(p.part_st + static_cast<size_t>(first + c) * 3 * 256 + prow_in_item);
          M = fmaxf(M, m_c[c]);
        }
      }
      float wl = 0.f, wr = 0.f;
#pragma unroll
      for (int c = 0; c < kMaxSplit; ++c) {
        w[c] = 0.f;
        if (c < k) {
          const float *st = p.part_st + static_cast<size_t>(first + c) * 3 * 256 + prow_in_item;
          const float e = ex2_approx(m_c[c] - M);
          wl += __ldcg(st + 256) * e;
          w[c] = __ldcg(st + 512) * e;
          wr += w[c];
        }
      }
      const float inv = 1.f / wr;
      const int q_idx = (it.qt0 + t) * 128 + row;
      const size_t row_off = static_cast<size_t>(it.bh) * p.N + q_idx;
      uint8_t *orow0 = reinterpret_cast<uint8_t *>(static_cast<uint16_t *>(p.o) +
                                                   (row_off - lane) * D + (D / 2) * hf);
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh) {  // 32 columns at a time
        float acc[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxSplit; ++c) {
          if (c < k) {
            const float wc = w[c] * inv;
            const float4 *src = p.part_o +
                                (static_cast<size_t>(first + c) * (D / 4) + (D / 8) * hf + 8 * hh) * 256 +
                                prow_in_item;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 x = __ldcg(src + u * 256);
              acc[4 * u] = fmaf(wc, x.x, acc[4 * u]);
              acc[4 * u + 1] = fmaf(wc, x.y, acc[4 * u + 1]);
              acc[4 * u + 2] = fmaf(wc, x.z, acc[4 * u + 2]);
              acc[4 * u + 3] = fmaf(wc, x.w, acc[4 * u + 3]);
            }
          }
        }
        uint4 v4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          v4[u] = make_uint4(pack2<BF16>(acc[8 * u], acc[8 * u + 1]),
                             pack2<BF16>(acc[8 * u + 2], acc[8 * u + 3]),
                             pack2<BF16>(acc[8 * u + 4], acc[8 * u + 5]),
                             pack2<BF16>(acc[8 * u + 6], acc[8 * u + 7]));
        store_rows<4>(v4, orow0 + 64 * hh, static_cast<size_t>(D) * 2,
                      p.N - (q_idx - static_cast<int>(lane)), lane);
      }
      if (q_idx < p.N && hf == 0) p.lse[row_off] = (M + lg2_approx(wl)) * 0.6931471805599453f;
    };
    const float sl2 = p.scale_log2;
    uint32_t st_need = 0, st_rows = 0, st_wres = 0, st_wblk = 0;  // STATS only
    uint32_t s_par = 0, o_par = 0, xpar = 0;  // barrier phase bits, exchange parity
    uint32_t pv_par = 0;                      // PV done phase bit (d = 64)
    // bar.sync cannot time out, so a warp whose wait gave up (ok == false)
    // keeps walking the same sequence of blocks, doing no work but taking
    // part in every pair barrier, so its partner can never be left waiting.
    bool ok = true;
    for (int round = 0; round * static_cast<int>(gridDim.x) < p.n_units; ++round) {
      const int item = round_item(round, p);
      if (item < 0) continue;
      const Item it = decode_unit(item, p);
      const int n = t ? it.n1 : it.n0;  // this tile's K/V blocks (0: no tile 1)
      // running max (log2 units), this half's sums of P and of P corrected
      // for the rounding of each block's largest value
      float m = -INFINITY, l = 0.f, r = 0.f;
      // epilogue: O / l to memory, logsumexp (one pair barrier on every
      // path, like a block)
      auto epilogue = [&]() {
        // O_t is complete after the tile's last PV (d = 64: its PV done)
        if constexpr (C::kSepP) {
          if (ok) ok = wait_bar(bar(C::kPVDone + t), pv_par, abort_flag, p.status);
          pv_par ^= 1u;
        } else {
          if (ok) ok = wait_bar(bar(C::kOFull + t), o_par, abort_flag, p.status);
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          pair_sync();
          return;
        }
        if constexpr (!C::kSepP) o_par ^= 1u;
        tc_fence_after();
        *xslot(xpar, hf, 0) = l;
        *xslot(xpar, hf, 1) = r;
        pair_sync();
        const float lsum = l + *xslot(xpar, hf ^ 1, 0);
        const float rsum = r + *xslot(xpar, hf ^ 1, 1);
        xpar ^= 1u;
        const float inv_l = 1.f / rsum;
        const uint64_t inv_l2 = f2(inv_l, inv_l);
        const int q_idx = (it.qt0 + t) * 128 + row;
        const bool live = q_idx < p.N;
        const size_t row_off = (static_cast<size_t>(it.bh) * p.N + q_idx);
        const uint32_t tO = t_lane + C::col_o(t) + (D / 2) * hf;
        if (it.piece >= 0) {
          // a piece of a split item: its O normalised by its own sum (fp32)
          // and its row statistics go to scratch memory for the merge, in a
          // column-group-major layout so that a warp's 32 rows are 512
          // contiguous bytes
          const int prow = t * 128 + row;
          float4 *dst = p.part_o + (static_cast<size_t>(it.piece) * (D / 4) + (D / 8) * hf) * 256 + prow;
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint32_t orr[32];
            tmem_ld32(tO + 32 * c, orr);
            tmem_ld_wait(orr);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              dst[(8 * c + u) * 256] = make_float4(__uint_as_float(orr[4 * u]) * inv_l,
                                                   __uint_as_float(orr[4 * u + 1]) * inv_l,
                                                   __uint_as_float(orr[4 * u + 2]) * inv_l,
                                                   __uint_as_float(orr[4 * u + 3]) * inv_l);
          }
          if (hf == 0) {
            float *st = p.part_st + static_cast<size_t>(it.piece) * 3 * 256 + prow;
            st[0] = m;
            st[256] = lsum;
            st[512] = rsum;
          }
          return;
        }
        // this warp's first row, its half of the columns; rows D * 2 bytes
        // apart; 32 columns (64 bytes of each row) at a time
        uint8_t *orow0 = reinterpret_cast<uint8_t *>(static_cast<uint16_t *>(p.o) +
                                                     (row_off - lane) * D + (D / 2) * hf);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t orr[32];
          tmem_ld32(tO + 32 * c, orr);
          tmem_ld_wait(orr);
          uint4 v4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float a, b;
              f2_split(fmul2(f2(__uint_as_float(orr[8 * u + 2 * e]),
                                __uint_as_float(orr[8 * u + 2 * e + 1])),
                             inv_l2),
                       a, b);
              w4[e] = pack2<BF16>(a, b);
            }
            v4[u] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
          store_rows<4>(v4, orow0 + 64 * c, static_cast<size_t>(D) * 2,
                        p.N - (q_idx - static_cast<int>(lane)), lane);
        }
        if (live && hf == 0)
          p.lse[row_off] = (m + lg2_approx(lsum)) * 0.6931471805599453f;
      };
      for (int j = 0; j < n; ++j) {
        {
          const int qt = it.qt0 + t;
          if (ok) ok = wait_bar(bar(C::kSFull + t), s_par, abort_flag, p.status);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) {  // failed: keep the pair barrier count in step, do nothing else
            pair_sync();
            continue;
          }
          s_par ^= 1u;
          tc_fence_after();
          const uint32_t tS = t_lane + C::col_s(t);
          uint32_t sr[2][32];
          tmem_ld32(tS + 64 * hf, sr[0]);
          tmem_ld32(tS + 64 * hf + 32, sr[1]);
          tmem_ld_wait(sr[0]);
          tmem_ld_wait(sr[1]);
          if constexpr (C::kSepP) {
            // S_t is in registers: the MMA may overwrite it with the next S
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kSFree + t));
          }
          float s[64];
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
          // mask only where needed: the diagonal block (causal) or the ragged
          // last block (non-causal, N % 128 != 0); c + 64h is the key column
          if (p.causal && j == qt) {
            const int lim = row - 64 * hf;
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c > lim) s[c] = -INFINITY;
          } else if (!p.causal && it.j0 + j == p.n_qtiles - 1 && (p.N & 127)) {
            const int lim = p.N - (it.j0 + j) * 128 - 64 * hf;
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c >= lim) s[c] = -INFINITY;
          }
          float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
          for (int c = 4; c < 60; c += 8) {
            mx[0] = fmax3(mx[0], s[c], s[c + 1]);
            mx[1] = fmax3(mx[1], s[c + 2], s[c + 3]);
            mx[2] = fmax3(mx[2], s[c + 4], s[c + 5]);
            mx[3] = fmax3(mx[3], s[c + 6], s[c + 7]);
          }
          mx[0] = fmax3(mx[0], s[60], s[61]);
          mx[1] = fmax3(mx[1], s[62], s[63]);
          const float hmax = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]);  // this half's max
          *xslot(xpar, hf, 0) = hmax;
          pair_sync();
          const float rmax = fmaxf(hmax, *xslot(xpar, hf ^ 1, 0));
          xpar ^= 1u;
          const float m_cand = fmaxf(m, rmax * sl2);
          const bool need = (m_cand - m) > p.rescale_thr;
          float alpha = 1.f;
          if (need) {
            alpha = ex2_approx(m - m_cand);
            m = m_cand;
          }
          if constexpr (C::kSepP) {
            // P_t and O_t are free once PV_t(j-1) is complete
            if (j > 0) {
              if (ok) ok = wait_bar(bar(C::kPVDone + t), pv_par, abort_flag, p.status);
              pv_par ^= 1u;
              ok = __all_sync(0xffffffffu, ok);
              tc_fence_after();
            }
          }
          // P = 2^(S*scale*log2e - m), rounded to the MMA's 16-bit type, over
          // the P columns [32h, 32h + 32) of this tile (keys 64h..64h+63).
          // Where P overlays S (d = 128), both warps have loaded their S
          // halves (the exchange above), so the P stores cannot overwrite S
          // the other warp still needs.
          const uint64_t sl2_2 = f2(sl2, sl2);
          const uint64_t negm_2 = f2(-m, -m);
          uint64_t sx2[2] = {0, 0};
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {  // two stores of 16 columns: fewer live registers
            uint32_t pk[16];
#pragma unroll
            for (int c = 32 * hh; c < 32 * hh + 32; c += 2) {
              const uint64_t x2 = ffma2(f2(s[c], s[c + 1]), sl2_2, negm_2);
              float e0, e1;
              if (C::kExpSplit > 0 && (c >> 1) % (C::kExpSplit > 0 ? C::kExpSplit : 1) ==
                                          C::kExpSplit - 1) {
                exp2_poly2<BF16>(x2, e0, e1);  // on the FMA pipes
              } else {
                float x0, x1;
                f2_split(x2, x0, x1);
                e0 = ex2_approx(x0);
                e1 = ex2_approx(x1);
              }
              pk[(c >> 1) & 15] = pack2<BF16>(e0, e1);
              sx2[(c >> 1) & 1] = fadd2(sx2[(c >> 1) & 1], f2(e0, e1));
            }
            tmem_st16(t_lane + C::col_p(t) + 32 * hf + 16 * hh, pk);
          }
          float sum_x, sum_r;
          {
            float a, b;
            f2_split(fadd2(sx2[0], sx2[1]), a, b);
            sum_x = a + b;
            sum_r = sum_x;
            if constexpr (BF16) {
              // O is normalised by the fp32 sum plus the rounding error of the
              // largest P of this half-block: in a peaked row the dominant
              // weight's rounding would otherwise reach O undivided, while the
              // other elements' rounding errors average out.  LSE uses the sum.
              const float top = ex2_approx(fmaf(hmax, sl2, -m));
              sum_r += __bfloat162float(__float2bfloat16_rn(top)) - top;
            }
          }
          l = l * alpha + sum_x;
          r = r * alpha + sum_r;
          // Conditional rescale of this half of the running output (v4
          // pseudo-code panel: "if need_rescale(m, m_new): acc *= exp(m -
          // m_new)").  PV_t(j-1) is complete -- its commit precedes S_t(j)'s
          // (d = 128), or its PV done was awaited above (d = 64) -- and
          // PV_t(j) waits for this block's signal.
          if constexpr (C::kStats) {
            if (j > 0) {
              if (hf == 0) {
                ++st_rows;
                st_need += need ? 1u : 0u;
              }
              if (lane == 0) ++st_wblk;
            }
          }
          if (j > 0 && __any_sync(0xffffffffu, need)) {
            if constexpr (C::kStats)
              if (lane == 0) ++st_wres;
            const uint32_t tO = t_lane + C::col_o(t) + (D / 2) * hf;
            const uint64_t alpha2 = f2(alpha, alpha);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {  // 32 columns at a time
              uint32_t orr[32];
              tmem_ld32(tO + 32 * c, orr);
              tmem_ld_wait(orr);
#pragma unroll
              for (int u = 0; u < 32; u += 2) {
                float a, b;
                f2_split(fmul2(f2(__uint_as_float(orr[u]), __uint_as_float(orr[u + 1])), alpha2),
                         a, b);
                orr[u] = __float_as_uint(a);
                orr[u + 1] = __float_as_uint(b);
              }
              tmem_st32(tO + 32 * c, orr);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::kPFull + t));
        }
      }
      if (n > 0) epilogue();
      if (it.piece >= 0) {
        // The piece's results are in scratch memory: make them visible to
        // the whole device, count the piece, and if it was the item's last
        // one, merge all pieces of the item.  The two barriers are taken on
        // every path.
        __threadfence();
        softmax_sync();
        if (threadIdx.x == 0) {
          unsigned last = 0;
          if (ok)
            last = atomicAdd(p.part_cnt + it.piece / p.split_k, 1u) ==
                   static_cast<unsigned>(p.split_k - 1);
          // acquire side of the count: the other pieces' scratch writes
          // (each fenced before its own count) are ordered before the
          // merge's reads
          if (last) __threadfence();
          *merge_flag = last;
        }
        softmax_sync();
        if (ok && *merge_flag && n > 0) merge(it, t);
      }
    }
    if constexpr (C::kStats) {
      unsigned long long v[4] = {st_need, st_rows, st_wres, st_wblk};  // widened once
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int sh = 16; sh >= 1; sh >>= 1) v[i] += __shfl_xor_sync(0xffffffffu, v[i], sh);
        if (lane == 0 && p.stats != nullptr) atomicAdd(p.stats + i, v[i]);
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Self-test of the failure path: one warp waits on a barrier that nothing
// ever arrives on.  The bounded wait must give up after `timeout_ns`, set
// the status word and return, leaving the context usable.
__global__ void fa_wait_selftest_kernel(unsigned *status, uint64_t timeout_ns, int *gave_up) {
  __shared__ __align__(8) uint64_t never;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&never), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const bool ok = wait_bar(smem_u32(&never), 0, &abort_flag, status, timeout_ns);
  if (threadIdx.x == 0) *gave_up = ok ? 0 : 1;
}

}  // namespace fa
