// fa_api.cu -- the C ABI declared in include/fa.h: argument checks, TMA
// tensor-map encoding, per-device state and the kernel launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "fa.h"
#include "fa_bwd_kernel.cuh"
#include "fa_kernel.cuh"

namespace {

__device__ unsigned g_fa_status = 0;  // per-device status word (FA_ERR_TIMEOUT source)
// fa_fwd_noalloc's scratch: a fixed array instead of pool memory
__device__ __align__(256) unsigned char g_fa_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
constexpr int kMaxVariants = 32;
constexpr int kOrderAuto = -2;  // causal item order: the library's choice

struct DeviceState {
  std::once_flag once;
  int err = FA_OK;  // FA_ERR_DEVICE / FA_ERR_CUDA if the device is unusable
  int dev = 0;
  int sm_count = 0;
  unsigned *status = nullptr;  // device address of g_fa_status
  std::once_flag pool_once;
  cudaMemPool_t pool = nullptr;  // stream-ordered scratch for split items (none: no split)
  uint8_t *noalloc = nullptr;    // device address of g_fa_noalloc_scratch
  // causal item order chosen per (B*H, Q tiles): the host simulation runs
  // once per shape
  std::mutex order_mu;
  std::unordered_map<uint64_t, int> order_cache;  // causal_order's result
  // encoded TMA tensor maps, direct-mapped by (address, shape, dtype): a map
  // depends on nothing else, so a hit needs no re-encoding
  struct MapEntry {
    const void *base = nullptr;
    int64_t BH = 0, N = 0, d = 0;
    bool bf16 = false, valid = false;
    CUtensorMap map;
  };
  static constexpr int kMapSlots = 64;
  std::mutex map_mu;
  MapEntry map_cache[kMapSlots];
  // fa_fwd_host: copy-in, compute and copy-out streams, events and device
  // staging memory (created on first use, staging grown as needed); calls
  // on one device take host_mu, so they run one at a time
  std::once_flag host_once;
  int host_err = FA_OK;
  std::mutex host_mu;
  cudaStream_t s_in = nullptr, s_cp = nullptr, s_out = nullptr;
  cudaEvent_t host_ev[3][3] = {};  // [slot][loaded, done, drained]
  uint8_t *stage = nullptr;
  size_t stage_bytes = 0;
  std::once_flag attr_once[kMaxVariants];  // shared-memory attribute, per kernel variant
  int attr_err[kMaxVariants] = {};
  std::once_flag bwd_attr_once[8];  // backward kernels: [d == 128][fp16][CTA pairs]
  int bwd_attr_err[8] = {};
};

DeviceState g_dev[kMaxDevices];
thread_local int t_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return FA_ERR_CUDA;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Bytes of the wave-tail split's scratch for `pieces` pieces of `items`
// items at head dim D: partial O (256 rows x D fp32 per piece), row
// statistics (3 x 256 fp32 per piece, rounded up to 256 bytes) and one
// counter per item.  Parts: [0] O, [1] statistics, [2] counters.
void split_scratch_bytes(size_t pieces, size_t items, int D, size_t part[3]) {
  part[0] = pieces * 256 * static_cast<size_t>(D) * sizeof(float);
  part[1] = (pieces * 256 * 3 * sizeof(float) + 255) & ~static_cast<size_t>(255);
  part[2] = items * sizeof(unsigned);
}

// The most any split plan needs on a device with G SMs: at most one piece
// per SM (R items x k pieces with k <= G / R) at the larger head dim.
size_t split_scratch_max(int G) {
  size_t part[3];
  split_scratch_bytes(static_cast<size_t>(G), static_cast<size_t>(G), 128, part);
  return part[0] + part[1] + part[2];
}

// Device checks once per device: compute capability 10.3 (the kernels are
// built for sm_103a only), SM count, device addresses of the status word
// and of fa_fwd_noalloc's fixed array.  Allocates no device memory.
int device_state(DeviceState **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_DEVICE;
  DeviceState &s = g_dev[dev];
  std::call_once(s.once, [&] {
    int major = 0, minor = 0;
    cudaError_t e1 = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaError_t e2 = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaError_t e3 = cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess) {
      t_last_cuda_error = static_cast<int>(e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3));
      s.err = FA_ERR_CUDA;
      return;
    }
    if (major != 10 || minor != 3) {
      s.err = FA_ERR_DEVICE;
      return;
    }
    void *addr = nullptr;
    cudaError_t e4 = cudaGetSymbolAddress(&addr, g_fa_status);
    if (e4 != cudaSuccess) {
      t_last_cuda_error = static_cast<int>(e4);
      s.err = FA_ERR_CUDA;
      return;
    }
    s.dev = dev;
    s.status = static_cast<unsigned *>(addr);
    void *scr = nullptr;
    cudaError_t e5 = cudaGetSymbolAddress(&scr, g_fa_noalloc_scratch);
    if (e5 != cudaSuccess) {
      t_last_cuda_error = static_cast<int>(e5);
      s.err = FA_ERR_CUDA;
      return;
    }
    s.noalloc = static_cast<uint8_t *>(scr);
  });
  if (s.err != FA_OK) return s.err;
  *out = &s;
  return FA_OK;
}

// The split-scratch pool of the device, created by the first call of an
// entry point that may use it (never by fa_fwd_noalloc): a private memory
// pool that keeps what it has allocated, filled at once with the largest
// scratch any call can need (taken and given back on a private stream), so
// that later calls issued one stream at a time make no device allocation.
// Without a pool the library runs every item whole; a failed reservation
// only leaves the pool to grow on first use.
void ensure_pool(DeviceState &s, int dev) {
  std::call_once(s.pool_once, [&] {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if (cudaMemPoolCreate(&s.pool, &props) != cudaSuccess) {
      s.pool = nullptr;
      cudaGetLastError();
      return;
    }
    uint64_t keep = UINT64_MAX;
    cudaMemPoolSetAttribute(s.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    cudaStream_t st = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) == cudaSuccess) {
      void *r = nullptr;
      if (cudaMallocFromPoolAsync(&r, split_scratch_max(s.sm_count), s.pool, st) == cudaSuccess)
        cudaFreeAsync(r, st);
      cudaStreamSynchronize(st);
      cudaStreamDestroy(st);
    }
    cudaGetLastError();
  });
}

// [B*H, N, d] view, box 128 rows x 64 columns, 128-byte swizzle; rows past
// N inside a box read as zero.
int make_map(CUtensorMap *m, const void *base, bool bf16, int64_t BH, int64_t N, int64_t d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return FA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * 2), static_cast<cuuint64_t>(N * d * 2)};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                  const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = static_cast<int>(r);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

// make_map through the device's cache of encoded maps.
int cached_map(DeviceState &ds, CUtensorMap *m, const void *base, bool bf16, int64_t BH, int64_t N,
               int64_t d) {
  uint64_t h = reinterpret_cast<uintptr_t>(base) >> 8;
  h = h * 0x9E3779B97F4A7C15ull ^ static_cast<uint64_t>(BH) * 0xC2B2AE3D27D4EB4Full ^
      static_cast<uint64_t>(N) * 0x165667B19E3779F9ull ^ static_cast<uint64_t>(d) ^
      (bf16 ? 1ull : 0ull);
  DeviceState::MapEntry &e = ds.map_cache[(h >> 32) % DeviceState::kMapSlots];
  {
    std::lock_guard<std::mutex> lock(ds.map_mu);
    if (e.valid && e.base == base && e.BH == BH && e.N == N && e.d == d && e.bf16 == bf16) {
      *m = e.map;
      return FA_OK;
    }
  }
  const int rc = make_map(m, base, bf16, BH, N, d);
  if (rc != FA_OK) return rc;
  std::lock_guard<std::mutex> lock(ds.map_mu);
  e.base = base;
  e.BH = BH;
  e.N = N;
  e.d = d;
  e.bf16 = bf16;
  e.map = *m;
  e.valid = true;
  return FA_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Causal item order.  In round r of the static schedule CTA b takes item
// r * G + b (even rounds) or r * G + G - 1 - b (odd rounds).  Taking the
// heaviest pairs first across all heads balances the SMs best, but once the
// heads' K/V outgrow L2 it reads a head's K/V from HBM again for each of its
// pairs; head by head (heaviest pair first within each head) keeps a head's
// K/V in L2 across its pairs, but leaves the last head's heavy pairs to end
// the launch.  So head by head takes its last g heads together, heaviest
// pair first across them (their K/V, at most 96 MiB, still fits in L2),
// with g chosen among a few sizes for the best balance.  The per-CTA load
// of each order is simulated (the larger tile's K/V blocks per item, plus
// about 1.3 blocks for the restart between items); head by head is taken
// unless it balances more than 8 percentage points worse than heaviest
// first across all heads: under the board's power limit the HBM re-reads
// cost clock speed, which outweighs a few points of balance.  Launches over
// 2^20 items keep the first order.  Returns -1 (heaviest first across all
// heads) or g >= 0 (head by head, g tail heads).
int causal_order(int BH, int n_qtiles, int n_pairs, int G, double kv_head_bytes) {
  const int64_t n = static_cast<int64_t>(BH) * n_pairs;
  if (n <= G || n > (int64_t(1) << 20)) return -1;
  // load of one item of each level (level 0 = the heaviest pair)
  std::vector<double> w(static_cast<size_t>(n_pairs));
  for (int level = 0; level < n_pairs; ++level) {
    const int qt1 = 2 * (n_pairs - 1 - level) + 1;
    w[static_cast<size_t>(level)] = (qt1 < n_qtiles ? qt1 + 1 : qt1) + 1.3;
  }
  std::vector<double> load(static_cast<size_t>(G));
  // g < 0: heaviest first across all heads; g >= 0: head by head, g tail heads
  auto balance = [&](int g) {
    std::fill(load.begin(), load.end(), 0.0);
    const int64_t first = g < 0 ? 0 : static_cast<int64_t>(BH - g) * n_pairs;
    const int width = g < 0 ? BH : g;  // heads taken together, level by level
    int level = 0, col = 0;            // of item i in the level-by-level part
    int hm_level = 0;                  // of item i in the head-by-head part
    int64_t i = 0;
    for (int64_t r = 0; i < n; ++r) {
      for (int off = 0; off < G && i < n; ++off, ++i) {
        int lv;
        if (i < first) {
          lv = hm_level;
          if (++hm_level == n_pairs) hm_level = 0;
        } else {
          lv = level;
          if (++col == width) {
            col = 0;
            ++level;
          }
        }
        load[static_cast<size_t>((r & 1) ? G - 1 - off : off)] += w[static_cast<size_t>(lv)];
      }
    }
    double sum = 0.0, mx = 0.0;
    for (double x : load) {
      sum += x;
      mx = std::max(mx, x);
    }
    return sum / G / mx;
  };
  int best_g = 0;
  double best = balance(0);
  for (int g : {2, 4, 6, 8, 12, 16, 24, 32}) {
    if (g >= BH || g * kv_head_bytes > 96.0 * 1024 * 1024) break;
    const double b = balance(g);
    if (b > best + 1e-9) {
      best = b;
      best_g = g;
    }
  }
  return best >= balance(-1) - 0.08 ? best_g : -1;
}

template <int D, bool BF16, int STAGES, int EXPSPLIT, bool STATS>
int launch(DeviceState &ds, int slot, const void *q, const void *k, const void *v, void *o,
           float *lse, int64_t BH, int64_t N, int causal, float scale, float thr, bool noalloc,
           unsigned long long *stats, int order, cudaStream_t stream) {
  using C = fa::Cfg<D, BF16, STAGES, EXPSPLIT, STATS>;
  auto kernel = fa::fa_fwd_kernel<D, BF16, STAGES, EXPSPLIT, STATS>;
  std::call_once(ds.attr_once[slot], [&] {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    ds.attr_err[slot] = static_cast<int>(e);
  });
  if (ds.attr_err[slot] != 0) return cuda_fail(static_cast<cudaError_t>(ds.attr_err[slot]));

  CUtensorMap tq, tk, tv;
  int rc;
  if ((rc = cached_map(ds, &tq, q, BF16, BH, N, D)) != FA_OK) return rc;
  if ((rc = cached_map(ds, &tk, k, BF16, BH, N, D)) != FA_OK) return rc;
  if ((rc = cached_map(ds, &tv, v, BF16, BH, N, D)) != FA_OK) return rc;

  fa::Params p;
  p.o = o;
  p.lse = lse;
  p.status = ds.status;
  p.N = static_cast<int>(N);
  p.BH = static_cast<int>(BH);
  p.n_qtiles = static_cast<int>((N + 127) / 128);
  p.n_pairs = (p.n_qtiles + 1) / 2;
  p.n_items = p.BH * p.n_pairs;
  p.causal = causal ? 1 : 0;
  // K and V of all heads beyond 64 MiB: L2 (126 MB) no longer holds them
  const double kv_bytes = 2.0 * static_cast<double>(BH) * static_cast<double>(N) * D * 2.0;
  p.causal_head_major = 0;
  p.causal_tail_heads = 0;
  if (causal && kv_bytes > 64.0 * 1024 * 1024) {
    const uint64_t key = (static_cast<uint64_t>(p.BH) << 32) | static_cast<uint32_t>(p.n_qtiles);
    std::lock_guard<std::mutex> lock(ds.order_mu);
    auto hit = ds.order_cache.find(key);
    if (hit == ds.order_cache.end()) {
      if (ds.order_cache.size() >= 4096) ds.order_cache.clear();  // bounded
      const int g = causal_order(p.BH, p.n_qtiles, p.n_pairs, ds.sm_count, kv_bytes / BH);
      hit = ds.order_cache.emplace(key, g).first;
    }
    p.causal_head_major = hit->second >= 0 ? 1 : 0;
    p.causal_tail_heads = hit->second >= 0 ? hit->second : 0;
  }
  if (causal && order != kOrderAuto) {  // fa_fwd_variant's override
    p.causal_head_major = order >= 0 ? 1 : 0;
    p.causal_tail_heads = order >= 0 ? order : 0;
  }
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.rescale_thr = thr;
  p.stats = stats;

  // Wave-tail split.  With G persistent CTAs, the last round holds
  // R = n_items mod G items and leaves G - R SMs idle; when R <= G / 2 each
  // of those items is cut into k = min(G / R, kMaxSplit, n_qtiles) pieces
  // along the keys, so the last round takes about 1/k of the time.  The
  // pieces' results go to scratch memory (stream-ordered, from the
  // library's pool; for fa_fwd_noalloc, the fixed array, and a plan that
  // does not fit it is rejected) and are merged by the last piece of each
  // item.
  p.n_units = p.n_items;
  p.split_first = p.n_items;
  p.split_k = 1;
  p.part_o = nullptr;
  p.part_st = nullptr;
  p.part_cnt = nullptr;
  void *scratch = nullptr;  // pool memory to give back after the launch
  if (!causal && (noalloc || ds.pool != nullptr)) {
    const int G = ds.sm_count;
    const int R = p.n_items % G;
    int k = R > 0 ? G / R : 0;
    if (k > fa::kMaxSplit) k = fa::kMaxSplit;
    if (k > p.n_qtiles) k = p.n_qtiles;
    if (k >= 2) {
      size_t part[3];
      split_scratch_bytes(static_cast<size_t>(R) * k, static_cast<size_t>(R), D, part);
      const size_t bytes_o = part[0], bytes_st = part[1], bytes_cnt = part[2];
      const size_t need = bytes_o + bytes_st + bytes_cnt;
      uint8_t *base = nullptr;
      // Under stream capture the scratch becomes a graph allocation
      // (cudaMallocAsync, freed by the graph behind the kernel) instead of
      // pool memory, so that capturing the call never breaks the capture.
      cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
      if (!noalloc && cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        cudaGetLastError();
        cap = cudaStreamCaptureStatusInvalidated;
      }
      if (noalloc) {
        if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH;
        base = ds.noalloc;
      } else if (cap == cudaStreamCaptureStatusActive) {
        if (cudaMallocAsync(&scratch, need, stream) == cudaSuccess)
          base = static_cast<uint8_t *>(scratch);
        else
          scratch = nullptr;  // the capture reports its own error
      } else if (cap != cudaStreamCaptureStatusNone) {
        // capture state unknown: run unsplit, touching no allocator
      } else if (cudaMallocFromPoolAsync(&scratch, need, ds.pool, stream) != cudaSuccess) {
        // a failed scratch allocation only means no split (its error is cleared)
        scratch = nullptr;
        cudaGetLastError();
      } else {
        base = static_cast<uint8_t *>(scratch);
      }
      if (base != nullptr) {
        if (cudaMemsetAsync(base + bytes_o + bytes_st, 0, bytes_cnt, stream) == cudaSuccess) {
          p.split_first = p.n_items - R;
          p.split_k = k;
          p.n_units = p.split_first + R * k;
          p.part_o = reinterpret_cast<float4 *>(base);
          p.part_st = reinterpret_cast<float *>(base + bytes_o);
          p.part_cnt = reinterpret_cast<unsigned *>(base + bytes_o + bytes_st);
        } else {
          cudaGetLastError();
          if (scratch != nullptr) cudaFreeAsync(scratch, stream);
          scratch = nullptr;
        }
      }
    }
  }

  const int grid = p.n_units < ds.sm_count ? p.n_units : ds.sm_count;
  // Programmatic dependent launch: the CTAs may be scheduled, and run
  // their prologue (barriers, tensor memory), while the previous kernel in
  // the stream drains; the kernel waits for that kernel's completion before
  // its first global memory access, so stream order holds for the data.
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(grid));
  lc.blockDim = dim3(C::kThreads);
  lc.dynamicSmemBytes = C::kSmemBytes;
  lc.stream = stream;
  cudaLaunchAttribute la[1];
  la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  la[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = la;
  lc.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&lc, kernel, tq, tk, tv, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (scratch != nullptr) cudaFreeAsync(scratch, stream);
  if (e != cudaSuccess) {
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
      return FA_ERR_DEVICE;
    return cuda_fail(e);
  }
  return FA_OK;
}

// Kernel variants built into the library.  The first entry of each (d,
// dtype) is the one the product entry points use; the others are the ring
// depths, exp splits and the rescale counter that fa_fwd_variant reaches
// for tuning and measurement.
typedef int (*LaunchFn)(DeviceState &, int, const void *, const void *, const void *, void *,
                        float *, int64_t, int64_t, int, float, float, bool,
                        unsigned long long *, int, cudaStream_t);
struct Variant {
  int d;
  bool bf16;
  int stages;     // K/V ring slots (the resolved count)
  int exp_split;  // every exp_split-th pair of exponentials on the FMA pipes (0: none)
  bool stats;
  LaunchFn fn;
};
#define FA_V(DD, BB, ST, SP, STATS) \
  Variant{DD, BB, fa::Cfg<DD, BB, ST, SP, STATS>::kStages, SP, STATS, launch<DD, BB, ST, SP, STATS>}
const Variant kVariants[] = {
    // defaults (product entry points)
    FA_V(64, true, 0, 0, false), FA_V(64, false, 0, 0, false),
    FA_V(128, true, 0, 0, false), FA_V(128, false, 0, 0, false),
    // d = 128 ring depths and exp splits
    FA_V(128, true, 2, 0, false), FA_V(128, true, 3, 0, false),
    FA_V(128, true, 0, 4, false), FA_V(128, true, 0, 2, false),
    FA_V(128, false, 3, 0, false),
    // d = 64 ring depths and exp splits
    FA_V(64, true, 4, 0, false), FA_V(64, true, 6, 0, false), FA_V(64, true, 10, 0, false),
    FA_V(64, true, 0, 4, false), FA_V(64, true, 0, 2, false),
    // rescale counters at the default configuration
    FA_V(64, true, 0, 0, true), FA_V(128, true, 0, 0, true), FA_V(128, false, 0, 0, true),
};
#undef FA_V
constexpr int kNumVariants = sizeof(kVariants) / sizeof(kVariants[0]);
static_assert(kNumVariants <= kMaxVariants, "more variants than per-device attribute slots");

// Index of the variant, or -1.  stages 0 = the default ring depth.
int find_variant(int d, bool bf16, int stages, int exp_split, bool stats) {
  for (int i = 0; i < kNumVariants; ++i) {
    const Variant &x = kVariants[i];
    const int def_stages = kVariants[(d == 64 ? 0 : 2) + (bf16 ? 0 : 1)].stages;
    if (x.d == d && x.bf16 == bf16 && x.stages == (stages ? stages : def_stages) &&
        x.exp_split == exp_split && x.stats == stats)
      return i;
  }
  return -1;
}

int fwd_common(bool bf16, const void *q, const void *k, const void *v, void *o, float *lse,
               int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
               float thr, fa_stream_t stream, bool noalloc = false, int variant = -1,
               unsigned long long *stats = nullptr, int order = kOrderAuto) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEADDIM;
  if (N > FA_MAX_N) return FA_ERR_UNSUPPORTED_N;
  // B*H*N*d elements (and the work-item count) must stay in range.
  const int64_t kLimit = int64_t(1) << 40;
  if (B > kLimit / H || B * H > kLimit / N || B * H * N > kLimit / d) return FA_ERR_SHAPE;
  const int64_t BH = B * H;
  if (BH * ((N + 255) / 256) > INT32_MAX / 2) return FA_ERR_SHAPE;
  for (const void *ptr : {q, k, v, static_cast<const void *>(o)})
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_ALIGN;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
  if (!(thr >= 0.f && thr <= FA_MAX_RESCALE_THRESHOLD)) return FA_ERR_OPTION;
  const size_t tbytes = static_cast<size_t>(BH * N * d) * 2;
  const size_t lbytes = static_cast<size_t>(BH * N) * 4;
  for (const void *in : {q, k, v})
    if (overlaps(o, tbytes, in, tbytes) || overlaps(lse, lbytes, in, tbytes)) return FA_ERR_ALIAS;
  if (overlaps(o, tbytes, lse, lbytes)) return FA_ERR_ALIAS;
  if (variant < 0) variant = (d == 64 ? 0 : 2) + (bf16 ? 0 : 1);  // the default variants
  if (kVariants[variant].d != d || kVariants[variant].bf16 != bf16) return FA_ERR_OPTION;
  if (order != kOrderAuto && (order < -1 || order > BH)) return FA_ERR_OPTION;

  DeviceState *ds = nullptr;
  int rc = device_state(&ds);
  if (rc != FA_OK) return rc;
  if (!noalloc) ensure_pool(*ds, ds->dev);
  return kVariants[variant].fn(*ds, variant, q, k, v, o, lse, BH, N, causal, scale, thr, noalloc,
                               stats, order, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------- backward
// Workspace of the backward: lse * log2(e) and D = rowsum(dO * O) per row,
// then the fp32 dQ accumulators, rows padded to whole 128-row tiles.
struct BwdWorkspace {
  size_t lse2 = 0, dd = 0, acc = 0, total = 0;  // byte offsets and size
};

BwdWorkspace bwd_workspace(int64_t BH, int64_t N, int64_t d) {
  const int64_t Np = (N + 127) / 128 * 128;
  BwdWorkspace w;
  w.lse2 = 0;
  w.dd = static_cast<size_t>(BH * Np) * 4;
  w.acc = w.dd + static_cast<size_t>(BH * Np) * 4;
  w.total = w.acc + static_cast<size_t>(BH * Np * d) * 4;
  return w;
}

int bwd_shape_check(int64_t B, int64_t H, int64_t N, int64_t d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEADDIM;
  if (N > FA_MAX_N) return FA_ERR_UNSUPPORTED_N;
  const int64_t kLimit = int64_t(1) << 40;
  if (B > kLimit / H || B * H > kLimit / N || B * H * N > kLimit / d) return FA_ERR_SHAPE;
  if (B * H * ((N + 127) / 128) > INT32_MAX / 2) return FA_ERR_SHAPE;
  return FA_OK;
}

// fa_bwd's kernel: one CTA per key block (false) or clusters of two that
// halve the dQ additions (true); fa_bwd_variant reaches both.
constexpr bool kBwdPairDefault = false;

template <int D, bool BF16, bool PAIR>
int launch_bwd(DeviceState &ds, const void *q, const void *k, const void *v, const void *o,
               const float *lse, const void *dout, void *dq, void *dk, void *dv,
               uint8_t *ws, int64_t BH, int64_t N, int causal, float scale, cudaStream_t stream) {
  using C = fa::BwdCfg<D, BF16>;
  auto kernel = fa::fa_bwd_kernel<D, BF16, PAIR>;
  const int slot = (D == 128 ? 4 : 0) + (BF16 ? 0 : 2) + (PAIR ? 1 : 0);
  std::call_once(ds.bwd_attr_once[slot], [&] {
    ds.bwd_attr_err[slot] = static_cast<int>(
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes));
  });
  if (ds.bwd_attr_err[slot] != 0) return cuda_fail(static_cast<cudaError_t>(ds.bwd_attr_err[slot]));
  CUtensorMap tq, tk, tv, tdo;
  int rc;
  if ((rc = cached_map(ds, &tq, q, BF16, BH, N, D)) != FA_OK) return rc;
  if ((rc = cached_map(ds, &tk, k, BF16, BH, N, D)) != FA_OK) return rc;
  if ((rc = cached_map(ds, &tv, v, BF16, BH, N, D)) != FA_OK) return rc;
  if ((rc = cached_map(ds, &tdo, dout, BF16, BH, N, D)) != FA_OK) return rc;
  const BwdWorkspace w = bwd_workspace(BH, N, D);
  fa::BwdParams p;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.lse2 = reinterpret_cast<float *>(ws + w.lse2);
  p.dd = reinterpret_cast<float *>(ws + w.dd);
  p.dq_acc = reinterpret_cast<float4 *>(ws + w.acc);
  p.status = ds.status;
  p.N = static_cast<int>(N);
  p.n_tiles = static_cast<int>((N + 127) / 128);
  p.Np = p.n_tiles * 128;
  p.BH = static_cast<int>(BH);
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  const dim3 tiles(static_cast<unsigned>(p.n_tiles), static_cast<unsigned>(BH));
  fa::fa_bwd_prep_kernel<D, BF16><<<tiles, 256, 0, stream>>>(p);
  cudaError_t e = cudaSuccess;
  if constexpr (PAIR) {
    // clusters of two CTAs over adjacent key blocks; an odd count of key
    // blocks per head gets one idle CTA to complete its last cluster
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(BH * (p.n_tiles + (p.n_tiles & 1))));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, tdo, p);
  } else {
    kernel<<<static_cast<unsigned>(BH * p.n_tiles), C::kThreads, C::kSmemBytes, stream>>>(
        tq, tk, tv, tdo, p);
  }
  if (e == cudaSuccess) fa::fa_bwd_dq_kernel<D, BF16><<<tiles, 128, 0, stream>>>(p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
      return FA_ERR_DEVICE;
    return cuda_fail(e);
  }
  return FA_OK;
}

int bwd_common(const void *q, const void *k, const void *v, const void *o, const float *lse,
               const void *dout, void *dq, void *dk, void *dv, void *workspace,
               size_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t d, int causal,
               float scale, int fp16, bool pair, fa_stream_t stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace)
    return FA_ERR_NULL;
  int rc = bwd_shape_check(B, H, N, d);
  if (rc != FA_OK) return rc;
  if (B * H > 65535) return FA_ERR_SHAPE;  // grid y of the row kernels
  for (const void *ptr : {q, k, v, o, dout, static_cast<const void *>(dq),
                          static_cast<const void *>(dk), static_cast<const void *>(dv)})
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGN;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
  const int64_t BH = B * H;
  const BwdWorkspace w = bwd_workspace(BH, N, d);
  if (workspace_bytes < w.total) return FA_ERR_WORKSPACE;
  const size_t tb = static_cast<size_t>(BH * N * d) * 2, lb = static_cast<size_t>(BH * N) * 4;
  const void *outs[3] = {dq, dk, dv};
  for (int a = 0; a < 3; ++a) {
    for (const void *in : {q, k, v, o, dout})
      if (overlaps(outs[a], tb, in, tb)) return FA_ERR_ALIAS;
    if (overlaps(outs[a], tb, lse, lb) || overlaps(outs[a], tb, workspace, w.total))
      return FA_ERR_ALIAS;
    for (int b = a + 1; b < 3; ++b)
      if (overlaps(outs[a], tb, outs[b], tb)) return FA_ERR_ALIAS;
  }
  for (const void *in : {q, k, v, o, dout})
    if (overlaps(workspace, w.total, in, tb)) return FA_ERR_ALIAS;
  if (overlaps(workspace, w.total, lse, lb)) return FA_ERR_ALIAS;

  DeviceState *ds = nullptr;
  rc = device_state(&ds);
  if (rc != FA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
#define FA_BWD(DD, BB, PP) launch_bwd<DD, BB, PP>(*ds, q, k, v, o, lse, dout, dq, dk, dv, ws, BH, N, causal, scale, st)
  if (pair) {
    if (d == 64) return fp16 ? FA_BWD(64, false, true) : FA_BWD(64, true, true);
    return fp16 ? FA_BWD(128, false, true) : FA_BWD(128, true, true);
  }
  if (d == 64) return fp16 ? FA_BWD(64, false, false) : FA_BWD(64, true, false);
  return fp16 ? FA_BWD(128, false, false) : FA_BWD(128, true, false);
#undef FA_BWD
}

}  // namespace

extern "C" {

int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
           int64_t H, int64_t N, int64_t d, int causal, float scale, fa_stream_t stream) {
  return fwd_common(true, q, k, v, o, lse, B, H, N, d, causal, scale,
                    FA_DEFAULT_RESCALE_THRESHOLD, stream);
}

int fa_fwd_fp16(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                int64_t H, int64_t N, int64_t d, int causal, float scale,
                fa_stream_t stream) {
  return fwd_common(false, q, k, v, o, lse, B, H, N, d, causal, scale,
                    FA_DEFAULT_RESCALE_THRESHOLD, stream);
}

int fa_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
              int64_t H, int64_t N, int64_t d, int causal, float scale, int fp16,
              float rescale_threshold, fa_stream_t stream) {
  return fwd_common(fp16 == 0, q, k, v, o, lse, B, H, N, d, causal, scale, rescale_threshold,
                    stream);
}

int fa_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                   int64_t H, int64_t N, int64_t d, int causal, float scale, int fp16,
                   float rescale_threshold, fa_stream_t stream) {
  return fwd_common(fp16 == 0, q, k, v, o, lse, B, H, N, d, causal, scale, rescale_threshold,
                    stream, /*noalloc=*/true);
}

int fa_fwd_variant(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                   int64_t H, int64_t N, int64_t d, int causal, float scale, int fp16,
                   float rescale_threshold, int stages, int exp_split, int causal_order,
                   unsigned long long *stats, fa_stream_t stream) {
  if (d != 64 && d != 128) return d < 1 ? FA_ERR_SHAPE : FA_ERR_HEADDIM;
  const int idx = find_variant(static_cast<int>(d), fp16 == 0, stages, exp_split, stats != nullptr);
  if (idx < 0) return FA_ERR_OPTION;
  if (stats != nullptr && (reinterpret_cast<uintptr_t>(stats) & 7u)) return FA_ERR_ALIGN;
  return fwd_common(fp16 == 0, q, k, v, o, lse, B, H, N, d, causal, scale, rescale_threshold,
                    stream, /*noalloc=*/false, idx, stats, causal_order);
}

int fa_bwd_workspace_size(int64_t B, int64_t H, int64_t N, int64_t d, size_t *bytes) {
  if (!bytes) return FA_ERR_NULL;
  const int rc = bwd_shape_check(B, H, N, d);
  if (rc != FA_OK) return rc;
  *bytes = bwd_workspace(B * H, N, d).total;
  return FA_OK;
}

int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, void *dq, void *dk, void *dv, void *workspace,
           size_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t d, int causal,
           float scale, int fp16, fa_stream_t stream) {
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H, N, d,
                    causal, scale, fp16, kBwdPairDefault, stream);
}

int fa_bwd_variant(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dout, void *dq, void *dk, void *dv, void *workspace,
                   size_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t d,
                   int causal, float scale, int fp16, int cta_pairs, fa_stream_t stream) {
  if (cta_pairs != 0 && cta_pairs != 1) return FA_ERR_OPTION;
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H, N, d,
                    causal, scale, fp16, cta_pairs == 1, stream);
}

int fa_variant_count(void) { return kNumVariants; }

int fa_causal_order(int64_t B, int64_t H, int64_t N, int64_t d, int sm_count) {
  if (B < 1 || H < 1 || N < 1 || N > FA_MAX_N || sm_count < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEADDIM;
  const int64_t BH = B * H;
  if (BH * ((N + 255) / 256) > INT32_MAX / 2) return FA_ERR_SHAPE;
  const int n_qtiles = static_cast<int>((N + 127) / 128), n_pairs = (n_qtiles + 1) / 2;
  const double kv_bytes = 2.0 * static_cast<double>(BH) * static_cast<double>(N) * d * 2.0;
  if (kv_bytes <= 64.0 * 1024 * 1024) return -1;
  return causal_order(static_cast<int>(BH), n_qtiles, n_pairs, sm_count, kv_bytes / BH);
}

int fa_variant_info(int index, int *d, int *fp16, int *stages, int *exp_split, int *stats) {
  if (index < 0 || index >= kNumVariants) return FA_ERR_OPTION;
  if (!d || !fp16 || !stages || !exp_split || !stats) return FA_ERR_NULL;
  const Variant &x = kVariants[index];
  *d = x.d;
  *fp16 = x.bf16 ? 0 : 1;
  *stages = x.stages;
  *exp_split = x.exp_split;
  *stats = x.stats ? 1 : 0;
  return FA_OK;
}

// Pipelined forward on host buffers: heads in chunks; chunk c+1 is copied
// in on s_in while chunk c is computed on s_cp and chunk c-1 is copied out on
// s_out, through `depth` rotating device staging buffers taken from the pool.
int fa_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                int64_t H, int64_t N, int64_t d, int causal, float scale, int fp16,
                int chunks) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEADDIM;
  if (N > FA_MAX_N) return FA_ERR_UNSUPPORTED_N;
  const int64_t kLimit = int64_t(1) << 40;
  if (B > kLimit / H || B * H > kLimit / N || B * H * N > kLimit / d) return FA_ERR_SHAPE;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
  if (chunks < 0 || chunks > FA_HOST_MAX_CHUNKS) return FA_ERR_OPTION;
  const int64_t BH = B * H;
  const size_t head_bytes = static_cast<size_t>(N * d) * 2, head_lse = static_cast<size_t>(N) * 4;
  const size_t tbytes = head_bytes * BH, lbytes = head_lse * BH;
  for (const void *in : {q, k, v})
    if (overlaps(o, tbytes, in, tbytes) || overlaps(lse, lbytes, in, tbytes)) return FA_ERR_ALIAS;
  if (overlaps(o, tbytes, lse, lbytes)) return FA_ERR_ALIAS;

  DeviceState *ds = nullptr;
  int rc = device_state(&ds);
  if (rc != FA_OK) return rc;
  std::call_once(ds->host_once, [&] {
    for (cudaStream_t *st : {&ds->s_in, &ds->s_cp, &ds->s_out}) {
      cudaError_t e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking);
      if (e != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(e);
        ds->host_err = FA_ERR_CUDA;
        return;
      }
    }
    for (int i = 0; i < 3; ++i)
      for (int j = 0; j < 3; ++j) {
        cudaError_t e = cudaEventCreateWithFlags(&ds->host_ev[i][j], cudaEventDisableTiming);
        if (e != cudaSuccess) {
          t_last_cuda_error = static_cast<int>(e);
          ds->host_err = FA_ERR_CUDA;
          return;
        }
      }
  });
  if (ds->host_err != FA_OK) return ds->host_err;
  std::lock_guard<std::mutex> lock(ds->host_mu);

  const int64_t nch = std::min<int64_t>(chunks == 0 ? FA_HOST_DEFAULT_CHUNKS : chunks, BH);
  int64_t width = 0;
  for (int64_t c = 0; c < nch; ++c)
    width = std::max(width, BH * (c + 1) / nch - BH * c / nch);
  const int depth = static_cast<int>(std::min<int64_t>(3, nch));
  // q, k, v, o, lse of one chunk; slots start on 256-byte boundaries
  const size_t slot_bytes = (4 * head_bytes * width + head_lse * width + 255) & ~size_t(255);
  cudaEvent_t(&ev)[3][3] = ds->host_ev;
  cudaError_t e = cudaSuccess;
  auto fail = [&](cudaError_t err) { rc = cuda_fail(err); };
  if (ds->stage_bytes < slot_bytes * depth) {  // grow the staging memory (all streams idle)
    if (ds->stage != nullptr) cudaFree(ds->stage);
    ds->stage = nullptr;
    ds->stage_bytes = 0;
    void *mem = nullptr;
    if ((e = cudaMalloc(&mem, slot_bytes * depth)) != cudaSuccess) return cuda_fail(e);
    ds->stage = static_cast<uint8_t *>(mem);
    ds->stage_bytes = slot_bytes * depth;
  }
  uint8_t *stage = ds->stage;
  const uint8_t *qh = static_cast<const uint8_t *>(q), *kh = static_cast<const uint8_t *>(k),
                *vh = static_cast<const uint8_t *>(v);
  uint8_t *oh = static_cast<uint8_t *>(o), *lh = reinterpret_cast<uint8_t *>(lse);
  for (int64_t c = 0; c < nch && rc == FA_OK; ++c) {
    const int64_t a = BH * c / nch, n = BH * (c + 1) / nch - a;
    const int i = static_cast<int>(c % depth);
    uint8_t *sq = stage + slot_bytes * i, *sk = sq + head_bytes * width,
            *sv = sk + head_bytes * width, *so = sv + head_bytes * width,
            *sl = so + head_bytes * width;
    const size_t tb = head_bytes * n, off = head_bytes * a;
    if (c >= depth && (e = cudaStreamWaitEvent(ds->s_in, ev[i][2], 0)) != cudaSuccess) { fail(e); break; }
    if ((e = cudaMemcpyAsync(sq, qh + off, tb, cudaMemcpyHostToDevice, ds->s_in)) != cudaSuccess ||
        (e = cudaMemcpyAsync(sk, kh + off, tb, cudaMemcpyHostToDevice, ds->s_in)) != cudaSuccess ||
        (e = cudaMemcpyAsync(sv, vh + off, tb, cudaMemcpyHostToDevice, ds->s_in)) != cudaSuccess ||
        (e = cudaEventRecord(ev[i][0], ds->s_in)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ds->s_cp, ev[i][0], 0)) != cudaSuccess) {
      fail(e);
      break;
    }
    rc = fwd_common(fp16 == 0, sq, sk, sv, so, reinterpret_cast<float *>(sl), n, 1, N, d, causal,
                    scale, FA_DEFAULT_RESCALE_THRESHOLD, ds->s_cp);
    if (rc != FA_OK) break;
    if ((e = cudaEventRecord(ev[i][1], ds->s_cp)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ds->s_out, ev[i][1], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(oh + off, so, tb, cudaMemcpyDeviceToHost, ds->s_out)) != cudaSuccess ||
        (e = cudaMemcpyAsync(lh + head_lse * a, sl, head_lse * n, cudaMemcpyDeviceToHost,
                             ds->s_out)) != cudaSuccess ||
        (e = cudaEventRecord(ev[i][2], ds->s_out)) != cudaSuccess) {
      fail(e);
      break;
    }
  }
  // s_out's last copy waits for the last forward, which waits for the last
  // copy in: on success that one stream covers all the work.  After a
  // failure part of the pipeline may not be chained, so all three are
  // drained before the staging memory can be reused.
  if (rc == FA_OK) {
    if ((e = cudaStreamSynchronize(ds->s_out)) != cudaSuccess) fail(e);
  } else {
    for (cudaStream_t st : {ds->s_in, ds->s_cp, ds->s_out}) cudaStreamSynchronize(st);
  }
  return rc;
}

int fa_selftest_wait_timeout(int64_t timeout_us, int *gave_up, fa_stream_t stream) {
  if (!gave_up) return FA_ERR_NULL;
  if (timeout_us < 1 || timeout_us > 1000000) return FA_ERR_OPTION;
  DeviceState *ds = nullptr;
  int rc = device_state(&ds);
  if (rc != FA_OK) return rc;
  fa::fa_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      ds->status, static_cast<uint64_t>(timeout_us) * 1000u, gave_up);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

int fa_get_status(fa_stream_t stream) {
  DeviceState *ds = nullptr;
  int rc = device_state(&ds);
  if (rc != FA_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned v = 0;
  e = cudaMemcpy(&v, ds->status, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (v != 0) {
    e = cudaMemset(ds->status, 0, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (v & fa::kStatusTimeout) return FA_ERR_TIMEOUT;
  return (v & fa::kStatusLayout) ? FA_ERR_INTERNAL : FA_OK;
}

const char *fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "success";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_SHAPE: return "B, H and N must be >= 1 and B*H*N*d must fit the index range";
    case FA_ERR_HEADDIM: return "head dimension d must be 64 or 128";
    case FA_ERR_UNSUPPORTED_N: return "sequence length N exceeds FA_MAX_N";
    case FA_ERR_ALIGN: return "q, k, v and o must be 16-byte aligned, lse 4-byte aligned";
    case FA_ERR_SCALE: return "scale must be finite and > 0";
    case FA_ERR_DEVICE: return "current device is not a compute capability 10.3 (sm_103a) GPU";
    case FA_ERR_CUDA: return "a CUDA runtime or driver call failed (see fa_last_cuda_error)";
    case FA_ERR_TIMEOUT: return "a pipeline wait inside the kernel gave up; outputs undefined";
    case FA_ERR_ALIAS: return "an output buffer overlaps an input or the other output";
    case FA_ERR_OPTION:
      return "option out of range (rescale_threshold in [0, FA_MAX_RESCALE_THRESHOLD], "
             "self-test limit in [1, 1e6] us)";
    case FA_ERR_SCRATCH:
      return "fa_fwd_noalloc: the split schedule needs more than FA_NOALLOC_SCRATCH_BYTES";
    case FA_ERR_WORKSPACE: return "fa_bwd: workspace smaller than fa_bwd_workspace_size";
    case FA_ERR_INTERNAL:
      return "a kernel found its shared memory base unaligned and did no work; outputs undefined";
    default: return "unknown error code";
  }
}

int fa_last_cuda_error(void) { return t_last_cuda_error; }

int fa_version(void) { return 100; }

}  // extern "C"
