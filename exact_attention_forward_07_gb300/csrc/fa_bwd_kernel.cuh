// fa_bwd_kernel.cuh -- the attention backward for sm_103a.
//
// Gradients of L = sum(dO * O) for the attention forward O = softmax(scale
// Q K^T [+ causal mask]) V, from the forward's O and logsumexp (the
// FlashAttention v4 Blackwell pipeline diagram names the backward pass in
// its pseudo-code panel, "backward idea", and its CTA-role panel: the
// backward accumulates dQ with atomic additions, which larger MMA tiles
// reduce).  With P recomputed from the logsumexp, per (query i, key j):
//
//   P  = exp(scale q_i.k_j - lse_i)           dV_j += P dO_i
//   dP = dO_i . v_j                           dS    = P (dP - D_i)
//   D_i = dO_i . O_i                          dQ_i += scale dS k_j
//                                             dK_j += scale dS q_i
//
// D_i = rowsum(dO * O) equals rowsum(P * dP) because O_i = sum_j P_ij v_j.
//
// Three kernels:
//   fa_bwd_prep_kernel   D and lse * log2(e) per row (padded to whole
//                        128-row tiles), and the dQ accumulators zeroed
//   fa_bwd_kernel        one CTA per (head, 128-key block j): K_j and V_j
//                        stay in shared memory while the CTA walks the
//                        query blocks i (causal: i >= j) through a two-stage
//                        TMA ring of Q_i and dO_i; five tcgen05 MMAs per step
//   fa_bwd_dq_kernel     dQ = scale * accumulators, rounded to 16 bits
//
// fa_bwd_kernel<PAIR = true> runs the same CTAs in clusters of two over
// adjacent key blocks, which exchange halves of each dQ product through
// distributed shared memory and so add half as many bytes to the fp32
// accumulators; the exchange ties the pair together on every step, and it
// is slower than the one-CTA kernel.
//
// Roles in fa_bwd_kernel (640 threads):
//   warp  0     TMA producer (one thread)
//   warp  1     MMA issue (one elected lane) + tensor-memory allocation
//   warps 4-19  compute warps: warp w owns lane quadrant w % 4 and a slice
//               of 32 columns; per step they form P^T and dS^T (one thread
//               per key), then read dQ out of tensor memory (one thread per
//               query row) and add it to the fp32 accumulators, half at once
//               and half spread over the next step's softmax; at the end
//               they write the block's dK and dV
//
// Per step (query block i):
//   S^T  = K_j Q_i^T      SS  -> TMEM [0,128)     (lanes = keys)
//   dP^T = V_j dO_i^T     SS  -> TMEM [128,256)
//   compute warps: P^T = 2^(S^T scale log2e - lse2_i), packed to 16 bits over
//   S^T; dS^T = P^T (dP^T - D_i) to shared memory, 128-byte swizzled; one
//   query half at a time
//   dV  += P^T dO_i       TS  (P^T from TMEM, dO_i MN-major), per query half
//   dK  += dS^T Q_i       SS  (dS^T K-major, Q_i MN-major), per query half
//   dQ_i = dS K_j         SS  (the same dS buffer read MN-major, K_j MN-major),
//                             between the two halves' dV and dK
// The dS buffer [query half][128 key rows][128 bytes] is at once the
// K-major layout of dS^T (rows = keys) and the MN-major layout of dS (64
// queries per swizzled row, keys along the rows), so one store serves both
// MMAs.  dQ goes to the columns of dP^T at d = 128 (tensor memory is full:
// S, dP, dK and dV take 512 columns), so the next dP^T waits until the
// compute warps have read it; at d = 64 it has columns of its own.
//
// Every wait is bounded as in the forward kernel; a wait that gives up sets
// the abort flag and the status word, in-flight copies and MMAs are drained
// and tensor memory is freed before the CTA exits.
#pragma once

#include "fa_kernel.cuh"

namespace fa {

constexpr uint32_t kStatusLayout = 2u;  // shared-memory base not 1024-byte aligned

struct BwdParams {
  const void *o;      // [BH, N, D] 16-bit forward output
  const void *dout;   // [BH, N, D] 16-bit
  const float *lse;   // [BH, N] natural-log logsumexp of the forward
  void *dq, *dk, *dv; // [BH, N, D] 16-bit
  float *lse2;        // [BH, Np]: lse * log2(e); +inf past N
  float *dd;          // [BH, Np]: rowsum(dO * O); 0 past N
  float4 *dq_acc;     // [BH][Np / 128][D / 4][128] fp32 x 4
  unsigned *status;
  int N, Np, BH;
  int n_tiles;        // Np / 128
  int causal;
  float scale;
  float scale_log2;   // scale * log2(e)
};

template <int D, bool BF16>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim must be 64 or 128");
  static constexpr int kTile = 128 * D * 2;   // one 128-row tile of 16-bit elements
  static constexpr int kHalf = 128 * 64 * 2;  // 64 columns of 128 rows: one swizzle span
  // depth of the Q/dO ring: at d = 64 the next step's first query half of
  // S^T and dP^T is issued one query half into the step, so its Q and dO
  // must be loaded a stage earlier; d = 128 has room for two
  static constexpr int kStages = D == 64 ? 3 : 2;
  static constexpr int kK = 0, kV = kTile;
  static constexpr int kQ = 2 * kTile;
  static constexpr int kDO = kQ + kStages * kTile;
  static constexpr int kDS = kDO + kStages * kTile;  // dS^T, [query half][128 key rows][128 bytes]
  static constexpr int kLse = kDS + 2 * kHalf;        // [stage][128] fp32
  static constexpr int kDd = kLse + kStages * 512;    // [stage][128] fp32
  static constexpr int kBar = kDd + kStages * 512;
  // barriers: K/V loaded; Q/dO stage full and empty (one each per stage); S^T and dP^T
  // done; dS written and dQ read (one arrival per compute warp each); dQ
  // done; dK/dV done; drain; for CTA pairs: the peer may write into this
  // CTA's dS buffer (arrived by the peer), the peer's dQ columns have landed
  // there (one local arrival + the bytes); and the first half of the query
  // columns' P^T and dS^T written (one arrival per compute warp); and (d =
  // 64) a step's second-half dV and dK done (an MMA commit), and S^T and
  // dP^T of the first query half done (bSdp then covers the second half)
  static constexpr int bKV = 0, bFull = 1, bEmpty = 1 + kStages, bSdp = 1 + 2 * kStages,
                       bDs = bSdp + 1, bDqFull = bSdp + 2, bDqFree = bSdp + 3, bDkdv = bSdp + 4,
                       bDrain = bSdp + 5, bSendOk = bSdp + 6, bRecv = bSdp + 7, bDsA = bSdp + 8,
                       bTail = bSdp + 9, bSdpA = bSdp + 10, kNumBars = bSdp + 11;
  static constexpr uint32_t kRecvBytes = 128 * (D / 2) * 4;  // half of dQ's columns, fp32
  static constexpr int kMisc = kBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kUsed = kMisc + 16;
  // 1 KiB of slack for the 1024-byte alignment of the tiles when it fits in
  // the 227 KiB a CTA may use; at d = 128 only 920 bytes fit, and the kernel
  // checks that the base it gets leaves room (it does when the dynamic
  // shared memory starts 1024-aligned)
  static constexpr int kMaxSmem = 227 * 1024;
  static constexpr int kSmemBytes = kUsed + 1024 < kMaxSmem ? kUsed + 1024 : kMaxSmem;
  static_assert(kUsed <= kMaxSmem, "shared memory beyond the per-CTA limit");
  static constexpr bool kDqAliasDp = (D == 128);
  static constexpr uint32_t cS = 0, cDP = 128, cDK = 256, cDV = 256 + D;
  static constexpr uint32_t cDQ = kDqAliasDp ? cDP : 256 + 2 * D;
  // d = 64: the second query half's P^T in columns of its own (the last
  // 64 are free), so the next step's S^T may overwrite S while it waits
  static constexpr uint32_t cP2 = 256 + 3 * D;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdescS = idesc_f16(BF16, false, 128, 128);         // S^T, dP^T
  static constexpr uint32_t kIdescSh = idesc_f16(BF16, false, 128, 64);          // one query half
  static constexpr uint32_t kIdescG = idesc_f16(BF16, true, 128, D);            // dV, dK
  static constexpr uint32_t kIdescQ = idesc_f16_ab(BF16, true, true, 128, D);   // dQ
  static constexpr int kThreads = 640;
  static constexpr int kComputeWarps = 16;
};

// D and lse * log2(e) for one 128-row tile of one head, and that tile's
// dQ accumulators zeroed.  256 threads; warp w takes rows 16w..16w+15, its
// lanes splitting each row's D columns.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const BwdParams p) {
  const int tile = blockIdx.x, bh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kPer = D / 32;  // elements per lane: 4 (d = 128) or 2 (d = 64)
  for (int r = 16 * warp; r < 16 * warp + 16; ++r) {
    const int n = tile * 128 + r;
    float dot = 0.f;
    if (n < p.N) {
      const size_t off = (static_cast<size_t>(bh) * p.N + n) * D + lane * kPer;
      const uint16_t *po = static_cast<const uint16_t *>(p.o) + off;
      const uint16_t *pd = static_cast<const uint16_t *>(p.dout) + off;
      uint16_t a[kPer], b[kPer];
      if constexpr (kPer == 4) {
        *reinterpret_cast<uint2 *>(a) = *reinterpret_cast<const uint2 *>(po);
        *reinterpret_cast<uint2 *>(b) = *reinterpret_cast<const uint2 *>(pd);
      } else {
        *reinterpret_cast<uint32_t *>(a) = *reinterpret_cast<const uint32_t *>(po);
        *reinterpret_cast<uint32_t *>(b) = *reinterpret_cast<const uint32_t *>(pd);
      }
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        float x, y;
        if constexpr (BF16) {
          x = __bfloat162float(__ushort_as_bfloat16(a[e]));
          y = __bfloat162float(__ushort_as_bfloat16(b[e]));
        } else {
          x = __half2float(__ushort_as_half(a[e]));
          y = __half2float(__ushort_as_half(b[e]));
        }
        dot = fmaf(x, y, dot);
      }
#pragma unroll
      for (int sh = 16; sh >= 1; sh >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, sh);
    }
    if (lane == 0) {
      const size_t row = static_cast<size_t>(bh) * p.Np + n;
      p.dd[row] = n < p.N ? dot : 0.f;
      p.lse2[row] = n < p.N ? p.lse[static_cast<size_t>(bh) * p.N + n] * 1.4426950408889634f
                            : INFINITY;
    }
  }
  float4 *acc = p.dq_acc + (static_cast<size_t>(bh) * p.n_tiles + tile) * (D / 4) * 128;
  for (int i = threadIdx.x; i < (D / 4) * 128; i += 256) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dQ = scale * accumulators, rounded to 16 bits: one 128-row tile of one
// head; thread = row, 32 columns at a time, stored through the in-warp
// transpose so each store instruction writes whole 64-byte row segments.
template <int D, bool BF16>
__global__ void __launch_bounds__(128) fa_bwd_dq_kernel(const BwdParams p) {
  const int tile = blockIdx.x, bh = blockIdx.y;
  const uint32_t lane = threadIdx.x & 31;
  const int row = threadIdx.x;
  const int n = tile * 128 + row;
  const float4 *acc =
      p.dq_acc + (static_cast<size_t>(bh) * p.n_tiles + tile) * (D / 4) * 128 + row;
  uint8_t *row0 = reinterpret_cast<uint8_t *>(static_cast<uint16_t *>(p.dq) +
                                              (static_cast<size_t>(bh) * p.N + n - lane) * D);
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint4 v4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 x = acc[(8 * c + 2 * u) * 128], y = acc[(8 * c + 2 * u + 1) * 128];
      v4[u] = make_uint4(pack2<BF16>(x.x * p.scale, x.y * p.scale),
                         pack2<BF16>(x.z * p.scale, x.w * p.scale),
                         pack2<BF16>(y.x * p.scale, y.y * p.scale),
                         pack2<BF16>(y.z * p.scale, y.w * p.scale));
    }
    store_rows<4>(v4, row0 + 64 * c, static_cast<size_t>(D) * 2, p.N - (n - static_cast<int>(lane)),
                  lane);
  }
}

// A compile-time bool as a value, for generic lambdas.
template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};

// NG groups of four fp32 additions: v[4u .. 4u + 3] into dst[128 u], the
// accumulator layout's float4 columns of one row.
template <int NG>
__device__ __forceinline__ void red_groups(float4 *dst, const uint32_t *v) {
#pragma unroll
  for (int u = 0; u < NG; ++u)
    red_add_v4(dst + u * 128, __uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
               __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
}

// Bounded wait on a barrier that the other CTA of the pair arrives on or
// writes through (acquire at cluster scope); false = give up.
__device__ __forceinline__ bool wait_bar_cl(uint32_t bar, uint32_t parity,
                                            volatile int *abort_flag, unsigned *status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        atomicOr(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// PAIR: CTAs run in clusters of two over adjacent key blocks 2c and 2c + 1
// of one head.  Both visit the same query blocks (causal: the even block's
// first, its diagonal, alone), and for each such block the pair halves its
// dQ additions: dQ_i = dS_i,2c K_2c + dS_i,2c+1 K_2c+1, so each CTA sends
// the peer the 16-column groups of its dQ product that the peer adds to
// L2 (st.async into the peer's dS buffer, free once the peer's dK and dQ
// MMAs have read it) and adds the peer's groups to its own before its
// reductions.  The pages' backward notes reach the same saving with two
// CTAs sharing one larger MMA tile.
template <int D, bool BF16, bool PAIR>
__global__ void __launch_bounds__(BwdCfg<D, BF16>::kThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
  using C = BwdCfg<D, BF16>;
  // d = 64 (one CTA per key block): steps overlap.  With the second query
  // half's P^T in its own tensor-memory columns, the next step's S^T and
  // dP^T go to the tensor core one query half at a time: the first half
  // once this step's first half of P^T and dS^T is formed (after this
  // step's first-half dV and dK), the second once dS is complete (ahead of
  // this step's dQ and second-half dV and dK).  The compute warps form the
  // next step's P^T and dS^T while those run, and read out this step's dQ
  // after that.
  constexpr bool kPipe = (D == 64) && !PAIR;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  if (sbase - raw + C::kUsed > static_cast<uint32_t>(C::kSmemBytes)) {
    // the tiles would not fit after alignment: every thread leaves at once
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  uint8_t *smem = smem_raw + (sbase - raw);
  const uint32_t bars = sbase + C::kBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_base_slot = reinterpret_cast<uint32_t *>(smem + C::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  // this CTA's key block; the CTAs of one head are consecutive, heaviest
  // (causal: the first key block sees every query block) first.  PAIR: an
  // odd count of key blocks is completed by an idle CTA, so that clusters
  // of two never straddle heads; the block before it works alone.
  const int T = p.n_tiles;
  const int Tg = PAIR ? T + (T & 1) : T;
  const int bh = blockIdx.x / Tg;
  const int jb = blockIdx.x - bh * Tg;
  const bool idle = PAIR && jb >= T;
  const uint32_t rank = PAIR ? static_cast<uint32_t>(jb & 1) : 0u;  // rank in the cluster
  const bool paired = PAIR && !idle && (jb ^ 1) < T;
  const int i0 = p.causal ? jb : 0;
  const int n_steps = idle ? 0 : T - i0;
  // first step whose query block the peer visits too
  const int xs0 = (p.causal && rank == 0) ? 1 : 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::bKV), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::bFull + s), 1);
      mbar_init(bar(C::bEmpty + s), 1);
    }
    mbar_init(bar(C::bSdp), 1);
    mbar_init(bar(C::bSdpA), 1);
    mbar_init(bar(C::bDs), C::kComputeWarps);      // one arrival per compute warp
    mbar_init(bar(C::bDsA), C::kComputeWarps);     // the same, first query half
    mbar_init(bar(C::bTail), 1);
    mbar_init(bar(C::bDqFull), 1);
    mbar_init(bar(C::bDqFree), C::kComputeWarps);  // one arrival per compute warp
    mbar_init(bar(C::bDkdv), 1);
    mbar_init(bar(C::bDrain), 1);
    mbar_init(bar(C::bSendOk), 1);  // the peer's one arrival per shared query block
    mbar_init(bar(C::bRecv), 1);    // this CTA's expect-bytes arrival
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_base_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;
  // the peer's barriers are initialised before either CTA signals the other
  if constexpr (PAIR) cluster_sync();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !idle) {
      const uint64_t pol_once = l2_policy_evict_first();  // K_j, V_j: read by this CTA only
      const uint64_t pol_reuse = l2_policy_evict_last();  // Q_i, dO_i: read by every CTA of the head
      mbar_arrive_expect_tx(bar(C::bKV), 2 * C::kTile);
      for (int h = 0; h < D / 64; ++h) {
        tma_load_3d(sbase + C::kK + h * C::kHalf, &tm_k, bar(C::bKV), h * 64, jb * 128, bh, pol_once);
        tma_load_3d(sbase + C::kV + h * C::kHalf, &tm_v, bar(C::bKV), h * 64, jb * 128, bh, pol_once);
      }
      int issued = 0;
      for (int t = 0; t < n_steps; ++t) {
        const int s = t % C::kStages;
        if (t >= C::kStages &&
            !wait_bar(bar(C::bEmpty + s), ((t / C::kStages) + 1) & 1u, abort_flag, p.status))
          break;
        const int i = i0 + t;
        mbar_arrive_expect_tx(bar(C::bFull + s), 2 * C::kTile + 1024);
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(sbase + C::kQ + s * C::kTile + h * C::kHalf, &tm_q, bar(C::bFull + s), h * 64,
                      i * 128, bh, pol_reuse);
          tma_load_3d(sbase + C::kDO + s * C::kTile + h * C::kHalf, &tm_do, bar(C::bFull + s),
                      h * 64, i * 128, bh, pol_reuse);
        }
        const size_t row = static_cast<size_t>(bh) * p.Np + static_cast<size_t>(i) * 128;
        bulk_load(sbase + C::kLse + s * 512, p.lse2 + row, 512, bar(C::bFull + s));
        bulk_load(sbase + C::kDd + s * 512, p.dd + row, 512, bar(C::bFull + s));
        ++issued;
      }
      // drain: every issued copy lands before shared memory is released
      wait_drain(bar(C::bKV), 0, abort_flag, p.status);
      for (int s = 0; s < C::kStages; ++s) {
        const int cnt = (issued - s + C::kStages - 1) / C::kStages;  // loads into stage s
        if (cnt > 0) wait_drain(bar(C::bFull + s), (cnt - 1) & 1u, abort_flag, p.status);
      }
    }
  } else if (warp == 1 && !idle) {
    // ------------------------------------------------------------- MMA issue
    const uint32_t leader = elect_one();
    const uint64_t kdesc0 = smem_desc_sw128(0, 16, 1024);       // K-major tiles
    const uint64_t mdesc0 = smem_desc_sw128(0, C::kHalf, 1024); // MN-major tiles
    // D[tmem] (+)= A B over a K extent of 16 * ksteps, A and B K-major tiles
    // of 64-column halves (the layout TMA writes)
    auto ss_kk = [&](uint32_t dcol, uint32_t a, uint32_t b, uint32_t idesc, int ksteps,
                     bool acc) {
      const uint64_t ad = kdesc0 + desc_addr(a), bd = kdesc0 + desc_addr(b);
      for (int kk = 0; kk < ksteps; ++kk) {
        const uint32_t off = ((kk >> 2) * C::kHalf + (kk & 3) * 32) >> 4;
        mma_ss_if(leader, tmem + dcol, ad + off, bd + off, idesc, (acc || kk > 0) ? 1u : 0u);
      }
    };
    bool ok = wait_bar(bar(C::bKV), 0, abort_flag, p.status);
    if constexpr (kPipe) {
      // S^T(t) and dP^T(t) of one query half h of a step (queries [64 h,
      // 64 h + 64): N = 64, B = rows 64 h.. of the Q and dO tiles, one
      // 128-byte row each at d = 64), once its Q and dO are loaded; the
      // first half's completion is bSdpA, the second's bSdp
      auto issue_sdp = [&](int tt, int h) -> bool {
        const int st = tt % C::kStages;
        if (h == 0) {
          if (!wait_bar(bar(C::bFull + st), (tt / C::kStages) & 1u, abort_flag, p.status))
            return false;
          tc_fence_after();
        }
        const uint32_t rows = static_cast<uint32_t>(h) * 64u * 128u;
        ss_kk(C::cS + 64 * h, sbase + C::kK, sbase + C::kQ + st * C::kTile + rows, C::kIdescSh,
              D / 16, false);
        ss_kk(C::cDP + 64 * h, sbase + C::kV, sbase + C::kDO + st * C::kTile + rows, C::kIdescSh,
              D / 16, false);
        mma_commit_if(leader, bar(h ? C::bSdp : C::bSdpA));
        return true;
      };
      if (ok && n_steps > 0) ok = issue_sdp(0, 0) && issue_sdp(0, 1);
      for (int t = 0; ok && t < n_steps; ++t) {
        const int s = t % C::kStages;
        const uint32_t q_s = sbase + C::kQ + s * C::kTile, do_s = sbase + C::kDO + s * C::kTile;
        const uint64_t bdo = mdesc0 + desc_addr(do_s), bq = mdesc0 + desc_addr(q_s);
        const uint64_t ads = kdesc0 + desc_addr(sbase + C::kDS);
        // first query half: P^T in S's columns
        if (!(ok = wait_bar(bar(C::bDsA), t & 1u, abort_flag, p.status))) break;
        tc_fence_after();
        for (int kk = 0; kk < 4; ++kk)
          mma_ts_if(leader, tmem + C::cDV, tmem + C::cS + 16 * kk, bdo + kk * (2048 >> 4),
                    C::kIdescG, (t > 0 || kk > 0) ? 1u : 0u);
        for (int kk = 0; kk < 4; ++kk)
          mma_ss_if(leader, tmem + C::cDK, ads + ((kk * 32) >> 4), bq + kk * (2048 >> 4),
                    C::kIdescG, (t > 0 || kk > 0) ? 1u : 0u);
        // the next step's first query half of S^T (its columns are free:
        // the first half's dV above read the P^T packed there) and dP^T
        // (read by this step's first half of the softmax)
        if (t + 1 < n_steps && !(ok = issue_sdp(t + 1, 0))) break;
        if (!(ok = wait_bar(bar(C::bDs), t & 1u, abort_flag, p.status))) break;
        tc_fence_after();
        // and its second half, read by this step's second half of the softmax
        if (t + 1 < n_steps && !(ok = issue_sdp(t + 1, 1))) break;
        if (t > 0) {  // dQ(t-1) read out of its columns
          if (!(ok = wait_bar(bar(C::bDqFree), (t - 1) & 1u, abort_flag, p.status))) break;
          tc_fence_after();
        }
        const uint64_t adt = mdesc0 + desc_addr(sbase + C::kDS);
        const uint64_t bk = mdesc0 + desc_addr(sbase + C::kK);
        for (int kk = 0; kk < 8; ++kk)
          mma_ss_if(leader, tmem + C::cDQ, adt + kk * (2048 >> 4), bk + kk * (2048 >> 4),
                    C::kIdescQ, kk > 0 ? 1u : 0u);
        mma_commit_if(leader, bar(C::bDqFull));
        // second query half: P^T in its own columns
        for (int kk = 4; kk < 8; ++kk)
          mma_ts_if(leader, tmem + C::cDV, tmem + C::cP2 + 8 * (kk - 4), bdo + kk * (2048 >> 4),
                    C::kIdescG, 1u);
        for (int kk = 4; kk < 8; ++kk)
          mma_ss_if(leader, tmem + C::cDK, ads + ((C::kHalf + (kk & 3) * 32) >> 4),
                    bq + kk * (2048 >> 4), C::kIdescG, 1u);
        mma_commit_if(leader, bar(C::bTail));       // its P^T columns and dS half free
        mma_commit_if(leader, bar(C::bEmpty + s));  // Q and dO of this stage read
      }
    } else {
    for (int t = 0; ok && t < n_steps; ++t) {
      const int s = t % C::kStages;
      const uint32_t q_s = sbase + C::kQ + s * C::kTile, do_s = sbase + C::kDO + s * C::kTile;
      if (!(ok = wait_bar(bar(C::bFull + s), (t / C::kStages) & 1u, abort_flag, p.status))) break;
      tc_fence_after();
      ss_kk(C::cS, sbase + C::kK, q_s, C::kIdescS, D / 16, false);     // S^T = K Q^T
      if (C::kDqAliasDp && t > 0) {  // dQ(t-1) read out of the dP columns
        if (!(ok = wait_bar(bar(C::bDqFree), (t - 1) & 1u, abort_flag, p.status))) break;
        tc_fence_after();
      }
      ss_kk(C::cDP, sbase + C::kV, do_s, C::kIdescS, D / 16, false);   // dP^T = V dO^T
      mma_commit_if(leader, bar(C::bSdp));
      // dV += P^T dO and dK += dS^T Q, K = the 128 queries, one half of them
      // at a time: the first half's products run while the compute warps
      // form the second half.  P^T of queries [16 kk, 16 kk + 16) is packed
      // in tensor-memory columns [16 kk, 16 kk + 8); dS^T is K-major in
      // shared memory; dO and Q are MN-major.
      const uint64_t bdo = mdesc0 + desc_addr(do_s), bq = mdesc0 + desc_addr(q_s);
      const uint64_t ads = kdesc0 + desc_addr(sbase + C::kDS);
      // dQ = dS K: the same buffer read MN-major, K MN-major.  It needs all
      // of dS, and goes first once dS is complete (before the second half
      // of dV and dK), so the compute warps' read-out of dQ and the next
      // step's dP^T start sooner.  The CTA pairs issue it last: their
      // "dQ done" must also mean that dK has finished reading dS.
      auto issue_dq = [&]() -> bool {
        if (!C::kDqAliasDp && t > 0) {  // dQ(t-1) read out of its own columns
          if (!wait_bar(bar(C::bDqFree), (t - 1) & 1u, abort_flag, p.status)) return false;
          tc_fence_after();
        }
        const uint64_t adt = mdesc0 + desc_addr(sbase + C::kDS);
        const uint64_t bk = mdesc0 + desc_addr(sbase + C::kK);
        for (int kk = 0; kk < 8; ++kk)
          mma_ss_if(leader, tmem + C::cDQ, adt + kk * (2048 >> 4), bk + kk * (2048 >> 4),
                    C::kIdescQ, kk > 0 ? 1u : 0u);
        mma_commit_if(leader, bar(C::bDqFull));
        return true;
      };
      for (int hq = 0; hq < 2 && ok; ++hq) {
        if (!(ok = wait_bar(bar(hq ? C::bDs : C::bDsA), t & 1u, abort_flag, p.status))) break;
        tc_fence_after();
        if (!PAIR && hq == 1 && !(ok = issue_dq())) break;
        for (int kk = 4 * hq; kk < 4 * hq + 4; ++kk)
          mma_ts_if(leader, tmem + C::cDV, tmem + C::cS + 16 * kk, bdo + kk * (2048 >> 4),
                    C::kIdescG, (t > 0 || kk > 0) ? 1u : 0u);
        for (int kk = 4 * hq; kk < 4 * hq + 4; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kHalf + (kk & 3) * 32) >> 4;
          mma_ss_if(leader, tmem + C::cDK, ads + off, bq + kk * (2048 >> 4), C::kIdescG,
                    (t > 0 || kk > 0) ? 1u : 0u);
        }
      }
      if (!ok) break;
      if (PAIR && !(ok = issue_dq())) break;
      mma_commit_if(leader, bar(C::bEmpty + s));  // Q and dO of this stage read
    }
    }
    if (ok) mma_commit_if(leader, bar(C::bDkdv));
    mma_commit_if(leader, bar(C::bDrain));
    wait_drain(bar(C::bDrain), 0, abort_flag, p.status);
  } else if (warp >= 4 && !idle) {
    // --------------------------------------------------------- compute warps
    // Sixteen warps; warp w owns the keys of lane quadrant w % 4 (one thread
    // per key) and the query columns [16 cs, 16 cs + 16) of each query half
    // (cs = (w - 4) / 4) of S^T, dP^T, P^T and dS^T, the first half before
    // the second, so that the first half's dV and dK products overlap the
    // second half's softmax; then a quarter of dQ's columns for the
    // query rows of its quadrant (32 at d = 128, 16 at d = 64; the CTA pairs
    // read 32 with warps cs < 2 at d = 64).  One pool of warps runs both
    // phases: at d = 128 the next dP^T waits for the dQ read-out, and at
    // d = 64 (kPipe) a step's dQ is read out after the next step's softmax.
    const int w = warp - 4;
    const int qd = w & 3, cs = w >> 2;
    const int row = qd * 32 + static_cast<int>(lane);  // key (phase 1) / query (phase 2)
    const bool key_dead = jb * 128 + row >= p.N;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(qd * 32) << 16);
    const uint64_t sl2_2 = f2(p.scale_log2, p.scale_log2);
    // PAIR: the peer's dS buffer and barriers, as seen from this CTA
    const uint32_t peer_buf = PAIR ? mapa_shared(sbase + C::kDS, rank ^ 1u) : 0u;
    const uint32_t peer_send_ok = PAIR ? mapa_shared(bar(C::bSendOk), rank ^ 1u) : 0u;
    const uint32_t peer_recv = PAIR ? mapa_shared(bar(C::bRecv), rank ^ 1u) : 0u;
    // dQ columns each warp reads out and adds: 32 (d = 128, and the CTA
    // pairs' exchange layout), or 16 at d = 64, where all sixteen warps then
    // share the read-out instead of eight.  Half of each step's additions
    // are deferred into the next step's softmax and spread over its eight
    // slots (sub-chunk x group of four query columns).  Issued all at once,
    // the additions fill the load/store queue and hold the warps past the
    // point where the next S^T and dP^T are ready (the chip takes fp32
    // additions at about twice the rate this kernel issued them); spread out
    // they drain while the exponentials run.
    constexpr int kQC = (PAIR || D == 128) ? 32 : D / 4;
    constexpr int kG = kQC / 4;  // their float4 groups
    constexpr int kDeferG = PAIR ? 0 : kG / 2;  // deferred float4 groups
    constexpr bool kDefer = kDeferG > 0;
    uint32_t pend[kDefer ? 4 * kDeferG : 1];
    float4 *pend_dst = nullptr;
    // Phase 2 of step tt: its dQ (query rows of this quadrant) into
    // registers; the tensor-memory columns are released before the
    // additions are issued, so the next MMAs overlap them.
    auto phase2 = [&](int tt) -> bool {
      const bool xchg = paired && tt >= xs0;
      const uint32_t xpar = static_cast<uint32_t>(tt - xs0) & 1u;
      bool ok = wait_bar(bar(C::bDqFull), tt & 1u, abort_flag, p.status);
      if (ok) {
      tc_fence_after();
      const int i = i0 + tt;
      if (PAIR && xchg && w == 0 && lane == 0) {
        // this CTA's dK and dQ MMAs have read its dS buffer: the peer may
        // write its columns there
        mbar_arrive_expect_tx(bar(C::bRecv), C::kRecvBytes);
        mbar_arrive_remote(peer_send_ok);
      }
      uint32_t r[kQC];
      if (kQC * cs < D) {
        if constexpr (kQC == 32) {
          tmem_ld32(t_lane + C::cDQ + kQC * cs, r);
        } else {
          tmem_ld16(t_lane + C::cDQ + kQC * cs, r);
        }
        tmem_ld_wait(r);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::bDqFree));
      if (kQC * cs < D) {
        float4 *dst = p.dq_acc + (static_cast<size_t>(bh) * T + i) * (D / 4) * 128 + row +
                      kG * cs * 128;
        if constexpr (PAIR) {
        if (xchg) {
          // columns 32 cs + 16 k + [0, 16) belong to rank k: send the
          // peer's sixteen, then add the peer's to this CTA's own
          uint32_t mine[16], theirs[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            mine[e] = rank ? r[16 + e] : r[e];
            theirs[e] = rank ? r[e] : r[16 + e];
          }
          ok = wait_bar_cl(bar(C::bSendOk), xpar, abort_flag, p.status);
          if (ok) {
#pragma unroll
            for (uint32_t u = 0; u < 4; ++u)
              st_async_v4(peer_buf + ((((4u * cs + u) << 7) + static_cast<uint32_t>(row)) << 4),
                          theirs[4 * u], theirs[4 * u + 1], theirs[4 * u + 2], theirs[4 * u + 3],
                          peer_recv);
            ok = wait_bar_cl(bar(C::bRecv), xpar, abort_flag, p.status);
          }
          if (ok) {
            const float4 *in = reinterpret_cast<const float4 *>(smem + C::kDS) + 4 * cs * 128 + row;
            float4 *dm = dst + 4 * rank * 128;
#pragma unroll
            for (uint32_t u = 0; u < 4; ++u) {
              const float4 x = in[u * 128];
              red_add_v4(dm + u * 128, __uint_as_float(mine[4 * u]) + x.x,
                         __uint_as_float(mine[4 * u + 1]) + x.y,
                         __uint_as_float(mine[4 * u + 2]) + x.z,
                         __uint_as_float(mine[4 * u + 3]) + x.w);
            }
          }
        } else {
          red_groups<kG>(dst, r);
        }
        } else if constexpr (kDefer) {
          red_groups<kG - kDeferG>(dst, r);
#pragma unroll
          for (int e = 0; e < 4 * kDeferG; ++e) pend[e] = r[4 * (kG - kDeferG) + e];
          pend_dst = dst;
        } else {
          red_groups<kG>(dst, r);
        }
      }
      }
      return ok;
    };
    bool ok = true;
    for (int t = 0; ok && t < n_steps; ++t) {
      // kPipe: each query half's S^T and dP^T has a barrier of its own
      ok = wait_bar(bar(kPipe ? C::bSdpA : C::bSdp), t & 1u, abort_flag, p.status);
      if (ok) {
      tc_fence_after();
      const int s = t % C::kStages, i = i0 + t;
      const float *lse2s = reinterpret_cast<const float *>(smem + C::kLse + s * 512);
      const float *dds = reinterpret_cast<const float *>(smem + C::kDd + s * 512);
      const bool diag = p.causal && i == jb;
      const bool masked = diag || (jb + 1) * 128 > p.N;
      // S^T and dP^T of this warp's 16 queries in the first query half; at
      // d = 64 (kPipe) the second half's are loaded while the first half's
      // P^T and dS^T are stored (at d = 128 that order measured 1 % slower)
      uint32_t sr[16], dr[16];
      tmem_ld16(t_lane + C::cS + 16 * cs, sr);
      tmem_ld16(t_lane + C::cDP + 16 * cs, dr);
      tmem_ld_wait(sr);
      tmem_ld_wait(dr);
#pragma unroll
      for (int sc = 0; sc < 2; ++sc) {
        const int q0 = 16 * cs + 64 * sc;  // first query column of this sub-chunk
        if (!kPipe && sc == 1) {
          tmem_ld16(t_lane + C::cS + q0, sr);
          tmem_ld16(t_lane + C::cDP + q0, dr);
          tmem_ld_wait(sr);
          tmem_ld_wait(dr);
        }
        uint32_t pk[8], gk[8];
        // P^T and dS^T of these 16 queries; MASK: the step needs the causal
        // diagonal or has keys past N (both uniform over the CTA), so the
        // other steps run without the per-element selects
        auto form = [&](auto mask_tag) {
          constexpr bool MASK = decltype(mask_tag)::value;
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            if constexpr (kDefer) {
              if (pend_dst != nullptr) {
#pragma unroll
                for (int k = 0; k < kDeferG; ++k)
                  if ((k * 8) / kDeferG == sc * 4 + e / 4)
                    red_groups<1>(pend_dst + (kG - kDeferG + k) * 128, pend + 4 * k);
              }
            }
            const float4 l4 = *reinterpret_cast<const float4 *>(lse2s + q0 + e);
            const float4 d4 = *reinterpret_cast<const float4 *>(dds + q0 + e);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
              float x0, x1;
              f2_split(ffma2(f2(__uint_as_float(sr[e + u]), __uint_as_float(sr[e + u + 1])), sl2_2,
                             f2(-lv[u], -lv[u + 1])),
                       x0, x1);
              float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              if constexpr (MASK) {
                if (key_dead || (diag && row > q0 + e + u)) p0 = 0.f;
                if (key_dead || (diag && row > q0 + e + u + 1)) p1 = 0.f;
              }
              float g0, g1;
              f2_split(fmul2(f2(p0, p1), fadd2(f2(__uint_as_float(dr[e + u]), __uint_as_float(dr[e + u + 1])),
                                               f2(-dv[u], -dv[u + 1]))),
                       g0, g1);
              pk[(e + u) >> 1] = pack2<BF16>(p0, p1);
              gk[(e + u) >> 1] = pack2<BF16>(g0, g1);
            }
          }
        };
        if (masked) {
          form(BoolTag<true>{});
        } else {
          form(BoolTag<false>{});
        }
        if (kPipe && sc == 0) {
          // the second half's S^T and dP^T have a barrier of their own
          if (!wait_bar(bar(C::bSdp), t & 1u, abort_flag, p.status)) ok = false;
          tc_fence_after();
          tmem_ld16(t_lane + C::cS + q0 + 64, sr);
          tmem_ld16(t_lane + C::cDP + q0 + 64, dr);
        }
        // kPipe: the previous step's dQ has read dS half 0 (and its
        // first-half dK before it), and its second-half dV and dK have read
        // P^T's own columns and dS half 1, before this step writes them
        if constexpr (kPipe) {
          if (t > 0 && !wait_bar(bar(sc ? C::bTail : C::bDqFull), (t - 1) & 1u, abort_flag,
                                 p.status))
            ok = false;
          tc_fence_after();
        }
        // P^T of these 16 queries: 8 packed columns over their own S^T
        // columns, already loaded (kPipe: the second half in its own columns)
        if (kDefer && sc == 1) pend_dst = nullptr;
        if (kPipe && sc == 1) {
          tmem_st8(t_lane + C::cP2 + 8 * cs, pk);
        } else {
          tmem_st8(t_lane + C::cS + q0, pk);
        }
        // dS^T: 32 bytes of the key's row in query half sc, 16-byte chunks
        // at their 128-byte-swizzle positions
        uint8_t *ds_row = smem + C::kDS + sc * C::kHalf + row * 128;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int pos = (2 * cs + u) ^ (row & 7);
          *reinterpret_cast<uint4 *>(ds_row + 16 * pos) =
              make_uint4(gk[4 * u], gk[4 * u + 1], gk[4 * u + 2], gk[4 * u + 3]);
        }
        if (sc == 0) {  // the first query half of P^T and dS^T is complete
          tmem_st_wait();
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::bDsA));
          if (kPipe) {
            tmem_ld_wait(sr);
            tmem_ld_wait(dr);
          }
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // dS^T stores visible to the tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::bDs));
      }
      if (ok) {
        if constexpr (kPipe) {
          if (t > 0) ok = phase2(t - 1);  // the previous step's dQ, read out behind this softmax
        } else {
          ok = phase2(t);
        }
      }
      // PAIR: no compute warp writes the next dS before all have read the
      // peer's columns out of the same buffer; taken on every step of a
      // paired CTA, so that a warp whose wait gave up leaves the loop at the
      // same step as all the others
      if (PAIR && paired) ok = bar_and(1, 32 * C::kComputeWarps, ok);
    }
    // the deferred additions still pending (those of the step before, for
    // the pipelined d = 64 path, whose phase 2 then runs the last time)
    if (kDefer && pend_dst != nullptr) red_groups<kDeferG>(pend_dst + (kG - kDeferG) * 128, pend);
    pend_dst = nullptr;
    if (kPipe && ok && n_steps > 0) ok = phase2(n_steps - 1);
    if (kDefer && pend_dst != nullptr) red_groups<kDeferG>(pend_dst + (kG - kDeferG) * 128, pend);
    // epilogue: dK (times scale) and dV of this quadrant's keys; 32 columns
    // each: d = 128, slice cs of both; d = 64, slices 0-1 take dK and 2-3 dV
    ok = __all_sync(0xffffffffu, ok);
    if (ok) ok = wait_bar(bar(C::bDkdv), 0, abort_flag, p.status);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const int key0 = jb * 128 + qd * 32;  // key of lane 0
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        int colx;  // first of the 32 columns this warp writes, or -1
        if constexpr (D == 128) {
          colx = 32 * cs;
        } else {
          colx = ((cs >> 1) == g) ? 32 * (cs & 1) : -1;
        }
        if (colx < 0) continue;
        uint8_t *row0 = reinterpret_cast<uint8_t *>(static_cast<uint16_t *>(g ? p.dv : p.dk) +
                                                    (static_cast<size_t>(bh) * p.N + key0) * D + colx);
        const float mul = g ? 1.f : p.scale;
        uint32_t r[32];
        tmem_ld32(t_lane + (g ? C::cDV : C::cDK) + colx, r);
        tmem_ld_wait(r);
        uint4 v4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          v4[u] = make_uint4(pack2<BF16>(__uint_as_float(r[8 * u]) * mul, __uint_as_float(r[8 * u + 1]) * mul),
                             pack2<BF16>(__uint_as_float(r[8 * u + 2]) * mul, __uint_as_float(r[8 * u + 3]) * mul),
                             pack2<BF16>(__uint_as_float(r[8 * u + 4]) * mul, __uint_as_float(r[8 * u + 5]) * mul),
                             pack2<BF16>(__uint_as_float(r[8 * u + 6]) * mul, __uint_as_float(r[8 * u + 7]) * mul));
        store_rows<4>(v4, row0, static_cast<size_t>(D) * 2, p.N - key0, lane);
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  // neither CTA of a pair leaves while the other may still signal it
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
