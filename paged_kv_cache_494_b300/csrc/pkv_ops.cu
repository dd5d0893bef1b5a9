// Device-operation entry points of libpagedkv (C ABI, see include/pagedkv.h): argument checks,
// launch planning, workspace layout and kernel dispatch. All device code lives in this
// translation unit (kernels_*.cuh are included here only).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cstdint>
#include <random>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <utility>

#include "kernels_cache.cuh"
#include "kernels_decode.cuh"
#include "kernels_prefill.cuh"
#include "kernels_prefill_tc.cuh"
#include "pkv_pool.hpp"

namespace pkv_dev {

// One warp waits on a fresh shared-memory mbarrier that nothing arrives on, with the bounded wait of
// the pipelined kernels: it gives up after kMaxPolls polls, records ERRBIT_TIMEOUT and returns.
// No copy or other asynchronous operation is in flight, so the block can exit at once.
__global__ void selftest_wait_kernel(int32_t* gave_up) {
  __shared__ __align__(8) uint64_t bar;
  set_error_word(nullptr);
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool done = mbar_wait_bounded(smem_addr(&bar), 0u);
  if (threadIdx.x == 0 && gave_up != nullptr) *gave_up = done ? 0 : 1;
}

}  // namespace pkv_dev

namespace {

using pkv_dev::DecodeArgs;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int num_sms() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cached[dev].store(v, std::memory_order_relaxed);
  return v;
}

// Programmatic dependent launch on every libpagedkv kernel unless PKV_PDL=0. Each kernel waits for
// its predecessor in the stream (griddepcontrol.wait) before touching global memory, so only the
// launch latency overlaps and data ordering is plain stream order; the one exception is the
// shared-prefix decode, whose decode kernel reads nothing its predecessor writes and waits for it
// only before completing (the tensor-core kernel lets it launch once its own inputs are complete).
bool pdl_enabled() {
  static const bool on = [] {
    const char* s = std::getenv("PKV_PDL");
    return !(s && std::strcmp(s, "0") == 0);
  }();
  return on;
}

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                   Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int env_int(const char* name, int fallback) {
  const char* s = std::getenv(name);
  if (!s || !*s) return fallback;
  const int v = std::atoi(s);
  return v > 0 ? v : fallback;
}

// ---------------------------------------------------------------------------------------------
// decode planning
// ---------------------------------------------------------------------------------------------
using DecodeKernel = void (*)(DecodeArgs, pkv_dev::TmaMaps);

enum MapKind { MAPS_NONE = 0, MAPS_BF16 = 1, MAPS_FP8 = 2 };

struct KernelPair {
  DecodeKernel decode = nullptr;
  DecodeKernel decode_defer = nullptr;   // the deferred-merge instantiation (bf16 pools only)
  int stage_bytes = 0;
  int maps = MAPS_NONE;   // which tensor maps the staging needs (1-D bulk copies when none)
};

template <class Math, int D, int G>
KernelPair pair_for(int maps) {
  KernelPair k;
  k.decode = pkv_dev::paged_decode_kernel<Math, D, G, false>;
  k.stage_bytes = Math::kStageBytes;
  k.maps = maps;
  return k;
}

template <int D, int G>
KernelPair pick_bf16(bool simt) {
  if (simt) {
    KernelPair k = pair_for<pkv_dev::SimtMath<__nv_bfloat16, D, G>, D, G>(MAPS_NONE);
    k.decode_defer = pkv_dev::paged_decode_kernel<pkv_dev::SimtMath<__nv_bfloat16, D, G>, D, G, true>;
    return k;
  }
  KernelPair k = pair_for<pkv_dev::MmaMath<D, G>, D, G>(MAPS_BF16);
  k.decode_defer = pkv_dev::paged_decode_kernel<pkv_dev::MmaMath<D, G>, D, G, true>;
  return k;
}

template <int D>
KernelPair pick_g(int dtype, int g, bool simt) {
  if (dtype == PKV_F32) {
    switch (g) {
      case 1: return pair_for<pkv_dev::SimtMath<float, D, 1>, D, 1>(MAPS_NONE);
      case 2: return pair_for<pkv_dev::SimtMath<float, D, 2>, D, 2>(MAPS_NONE);
      case 3: return pair_for<pkv_dev::SimtMath<float, D, 3>, D, 3>(MAPS_NONE);
      case 4: return pair_for<pkv_dev::SimtMath<float, D, 4>, D, 4>(MAPS_NONE);
      case 5: return pair_for<pkv_dev::SimtMath<float, D, 5>, D, 5>(MAPS_NONE);
      case 6: return pair_for<pkv_dev::SimtMath<float, D, 6>, D, 6>(MAPS_NONE);
      case 8: return pair_for<pkv_dev::SimtMath<float, D, 8>, D, 8>(MAPS_NONE);
      default: return KernelPair{};
    }
  }
  switch (g) {
    case 1: return pick_bf16<D, 1>(simt);
    case 2: return pick_bf16<D, 2>(simt);
    case 3: return pick_bf16<D, 3>(simt);
    case 4: return pick_bf16<D, 4>(simt);
    case 5: return pick_bf16<D, 5>(simt);
    case 6: return pick_bf16<D, 6>(simt);
    case 7: return pick_bf16<D, 7>(simt);
    case 8: return pick_bf16<D, 8>(simt);
    default: return KernelPair{};
  }
}

// tcgen05 prefill kernels: two Q tiles per CTA (one CTA per SM) sharing a 4-stage ring of 64-key steps.
constexpr int kTcTiles = 2, kTcStages = 4;
struct TcKernel {
  void (*kern)(pkv_dev::PrefillArgs, pkv_dev::TcMaps) = nullptr;
  size_t smem = 0;
  int item = 0;      // query tokens per CTA
  int threads = 0;
};
template <int D, int G, int NT, int ST>
TcKernel tc_pick(int32_t n_seqs) {
  using Sh = pkv_dev::TcShape<D, G, NT, ST>;
  TcKernel k;
  k.kern = pkv_dev::paged_prefill_tc_kernel<D, G, NT, ST>;
  k.smem = pkv_dev::prefill_tc_smem_bytes<Sh>(n_seqs);
  k.item = NT * Sh::TQ;
  k.threads = Sh::THREADS;
  return k;
}

// Prefill runs on the tcgen05 kernel unless PKV_PREFILL_PATH=mma (the mma.sync kernel, kept to
// cross-check the two) or the batch has more sequences than the tcgen05 kernel keeps in shared memory.
constexpr int32_t kPrefillTcMaxSeqs = 2048;
bool prefill_path_tc() {
  const char* s = std::getenv("PKV_PREFILL_PATH");
  return !(s && std::strcmp(s, "mma") == 0);
}

// PKV_DECODE_PATH=simt selects the CUDA-core path for bf16 as well (used to cross-check paths).
bool force_simt() {
  const char* s = std::getenv("PKV_DECODE_PATH");
  return s && std::strcmp(s, "simt") == 0;
}

KernelPair pick_fp8(int g) {
  // PKV_DECODE_FP8_CTAS=4: the G = 4 fp8 kernel compiled for 4 resident CTAs per SM (128 registers)
  if (g == 4 && env_int("PKV_DECODE_FP8_CTAS", 3) == 4) return pair_for<pkv_dev::Fp8Math<4, 4>, 128, 4>(MAPS_FP8);
  switch (g) {
    case 1: return pair_for<pkv_dev::Fp8Math<1>, 128, 1>(MAPS_FP8);
    case 2: return pair_for<pkv_dev::Fp8Math<2>, 128, 2>(MAPS_FP8);
    case 3: return pair_for<pkv_dev::Fp8Math<3>, 128, 3>(MAPS_FP8);
    case 4: return pair_for<pkv_dev::Fp8Math<4>, 128, 4>(MAPS_FP8);
    case 5: return pair_for<pkv_dev::Fp8Math<5>, 128, 5>(MAPS_FP8);
    case 6: return pair_for<pkv_dev::Fp8Math<6>, 128, 6>(MAPS_FP8);
    case 7: return pair_for<pkv_dev::Fp8Math<7>, 128, 7>(MAPS_FP8);
    case 8: return pair_for<pkv_dev::Fp8Math<8>, 128, 8>(MAPS_FP8);
    default: return KernelPair{};
  }
}

KernelPair pick_kernels(int dtype, int D, int g) {
  if (dtype == PKV_FP8) return D == 128 ? pick_fp8(g) : KernelPair{};
  if (dtype != PKV_F32 && dtype != PKV_BF16) return KernelPair{};
  const bool simt = force_simt();
  if (dtype == PKV_F32 && g == 7) return KernelPair{};
  if (D == 64) return pick_g<64>(dtype, g, simt);
  if (D == 128) return pick_g<128>(dtype, g, simt);
  return KernelPair{};
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// One cache tensor viewed as a 2-D bf16 array [NB*Hkv*B rows][D], boxes of 16 rows x 64 elements
// (128 bytes), 128-byte swizzle.
bool encode_cache_map(CUtensorMap* m, const void* base, const pkv_pool_desc& d) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d.head_dim),
                        static_cast<cuuint64_t>(d.num_blocks) * d.num_kv_heads * d.block_size};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d.head_dim) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(pkv_dev::kChunk)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 pools with head_dim 128, for the decode: the [rows][128] array viewed as 3-D (64 dims, rows,
// the two 128-byte halves of a row; the halves' stride, 128 bytes, is the outer one), boxes of
// 64 x 16 x 2 with 128-byte swizzle: one copy brings a chunk's K (or V) as the two boxes of the 2-D
// map, half after half.
bool encode_cache_map_halves(CUtensorMap* m, const void* base, const pkv_pool_desc& d) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || d.head_dim != 128) return false;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(d.num_blocks) * d.num_kv_heads * d.block_size, 2};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d.head_dim) * 2, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(pkv_dev::kChunk), 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp8 pools: K codes as a 2-D uint8 [NB*Hkv*B rows][D] array (boxes of 16 rows x 128 bytes, 128-byte
// swizzle); V codes as a 2-D uint8 [NB*Hkv*D rows][B] array (dim-major pages; boxes of 128 rows x
// 16 bytes, no swizzle).
bool encode_fp8_maps(pkv_dev::TmaMaps* maps, const void* k_cache, const void* v_cache, const pkv_pool_desc& d) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || d.head_dim != 128) return false;
  cuuint32_t estr[2] = {1, 1};
  cuuint64_t kdims[2] = {static_cast<cuuint64_t>(d.head_dim),
                         static_cast<cuuint64_t>(d.num_blocks) * d.num_kv_heads * d.block_size};
  cuuint64_t kstr[1] = {static_cast<cuuint64_t>(d.head_dim)};
  cuuint32_t kbox[2] = {128, static_cast<cuuint32_t>(pkv_dev::kChunk)};
  if (fn(&maps->k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(k_cache), kdims, kstr, kbox, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cuuint64_t vdims[2] = {static_cast<cuuint64_t>(d.block_size),
                         static_cast<cuuint64_t>(d.num_blocks) * d.num_kv_heads * d.head_dim};
  cuuint64_t vstr[1] = {static_cast<cuuint64_t>(d.block_size)};
  cuuint32_t vbox[2] = {static_cast<cuuint32_t>(pkv_dev::kChunk), static_cast<cuuint32_t>(d.head_dim)};
  return fn(&maps->v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(v_cache), vdims, vstr, vbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q of a prefill call as a 3-D bf16 array [total_q][Hq][D], boxes of (128 / G) tokens x G heads x 64
// dims with 128-byte swizzle: one box lands as the rows (token, head of the group) of a Q tile.
bool encode_q_map(CUtensorMap* m, const void* q, int32_t total_q, int32_t Hq, int32_t D, int32_t G) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(total_q)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hq) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(pkv_dev::kTcRows / G)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raises a kernel's dynamic shared-memory limit once per (kernel, device, size).
bool ensure_smem(const void* fn, size_t bytes) {
  static std::mutex mu;
  static std::unordered_map<const void*, size_t> done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done[dev].find(fn);
  if (it != done[dev].end() && it->second >= bytes) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) != cudaSuccess)
    return false;
  done[dev][fn] = bytes;
  return true;
}

// Resident CTAs per SM of a kernel at a block size and dynamic shared-memory size, looked up once
// per (device, kernel, block, smem): the occupancy query is the costliest host step of a launch.
int occupancy(const void* fn, int threads, size_t smem) {
  struct Key {
    int dev;
    const void* fn;
    int threads;
    size_t smem;
    bool operator==(const Key& o) const { return dev == o.dev && fn == o.fn && threads == o.threads && smem == o.smem; }
  };
  struct KeyHash {
    size_t operator()(const Key& k) const {
      return std::hash<const void*>()(k.fn) ^ (static_cast<size_t>(k.dev) << 48) ^
             (static_cast<size_t>(k.threads) << 32) ^ k.smem;
    }
  };
  static std::mutex mu;
  static std::unordered_map<Key, int, KeyHash> cache;
  Key key{0, fn, threads, smem};
  if (cudaGetDevice(&key.dev) != cudaSuccess) return 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = per_sm;
  return per_sm;
}

// Launches the tcgen05 prefill kernel for the arguments in `a` (items: NT Q tiles of 128 / G tokens;
// shared-prefix mode when a.shared_len > 0). grid_items: number of work items when known, else -1.
pkv_status tc_prefill_launch(const pkv_pool* p, const pkv_dev::PrefillArgs& a, const void* k_cache,
                             const void* v_cache, cudaStream_t st, int64_t grid_items) {
  const pkv_pool_desc& d = p->desc;
  const int g = a.Hq / d.num_kv_heads;
  TcKernel tk;
#define PKV_TC_CASE(DD, GG) \
  if (d.head_dim == DD && g == GG) tk = tc_pick<DD, GG, kTcTiles, kTcStages>(a.n_seqs);
  PKV_TC_CASE(64, 1) PKV_TC_CASE(64, 2) PKV_TC_CASE(64, 3) PKV_TC_CASE(64, 4)
  PKV_TC_CASE(64, 5) PKV_TC_CASE(64, 6) PKV_TC_CASE(64, 7) PKV_TC_CASE(64, 8)
  PKV_TC_CASE(128, 1) PKV_TC_CASE(128, 2) PKV_TC_CASE(128, 3) PKV_TC_CASE(128, 4)
  PKV_TC_CASE(128, 5) PKV_TC_CASE(128, 6) PKV_TC_CASE(128, 7) PKV_TC_CASE(128, 8)
#undef PKV_TC_CASE
  if (!tk.kern) return PKV_ERR_INVALID;
  if (!ensure_smem(reinterpret_cast<const void*>(tk.kern), tk.smem)) return PKV_ERR_CUDA;
  pkv_dev::TcMaps maps;
  std::memset(&maps, 0, sizeof maps);
  if (!encode_cache_map(&maps.k, k_cache, d) || !encode_cache_map(&maps.v, v_cache, d) ||
      !encode_q_map(&maps.q, a.q, a.total_q, a.Hq, d.head_dim, g))
    return PKV_ERR_CUDA;
  // persistent: one CTA per SM (or fewer when there are fewer work items)
  const int64_t items_ub = grid_items >= 0 ? grid_items
                                           : ((static_cast<int64_t>(a.total_q) + tk.item - 1) / tk.item + a.n_seqs) *
                                                 d.num_kv_heads;
  const int sms = num_sms();
  if (sms <= 0) return PKV_ERR_CUDA;
  const unsigned grid = static_cast<unsigned>(items_ub < sms ? (items_ub > 0 ? items_ub : 1) : sms);
  if (launch(tk.kern, dim3(grid), dim3(tk.threads), tk.smem, st, a, maps) != cudaSuccess ||
      cudaGetLastError() != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

// Query tokens per tcgen05 prefill work item for a head dimension and group size (0 if unsupported).
int tc_item_tokens(int D, int g) {
  if ((D != 64 && D != 128) || g < 1 || g > 8) return 0;
  return kTcTiles * (pkv_dev::kTcRows / g);
}

struct DecodePlan {
  KernelPair k;
  int nw = 4, stages = 2, grid = 0, warps = 0, max_tasks = 0;
  size_t smem = 0;
  int part_chunks = 0, max_parts = 0;
  int64_t n_units = 0, n_slots = 0;
  size_t off_ml = 0, off_o = 0, off_meta = 0, ws_bytes = 0;
  bool defer = false;
};

// Deferred-merge decode (dynamic tasks, then the merge kernel) for pkv_paged_decode(_window, _fp8)
// when PKV_DECODE_DEFER=1; otherwise the in-kernel merge. Measured on B300 (same box, L2 flushed):
// balanced split, deferred is slower (every task pays its own setup: locate, length and query loads,
// which a static range pays once per unit): serving batch 0.826 against 0.868 of the copy bandwidth,
// 8 x 32k tokens 248 against 210 us; 512-token partitions, it wins on long contexts (8 x 32k: 217 against
// 223-228 us) and loses on medium ones (64 sequences, G 5: 72 against 64 us; 128 children of a shared
// prompt: 101 against 90 us); the host does not know the lengths, so the default stays in-kernel. The
// shared-prefix decode always uses it: its merge kernel runs anyway and its decode starts beside another
// kernel.
bool decode_defer_wanted(int32_t) { return env_int("PKV_DECODE_DEFER", 0) > 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Tag of a decode call for the workspace's arrival counters: 48 bits, odd (so never the zero of fresh
// memory) and distinct for 2^47 consecutive calls of the process (2 * counter + 1, the counter
// started at a random point), so counts left by earlier calls are never taken for this call's.
unsigned long long next_call_tag() {
  static std::atomic<unsigned long long> counter{[] {
    std::random_device rd;
    return (static_cast<unsigned long long>(rd()) << 20) ^
           static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count());
  }()};
  return ((counter.fetch_add(1, std::memory_order_relaxed) << 1) | 1ull) & 0xffffffffffffull;
}

// Largest dynamic shared memory one block may opt into on the current device (cached per device).
size_t max_smem_optin() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v > 0) return static_cast<size_t>(v);
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  cached[dev].store(v, std::memory_order_relaxed);
  return static_cast<size_t>(v);
}

// defer: the deferred-merge mode (dynamic tasks, 2 slots per task, up to 4 tasks per warp).
pkv_status plan_decode(const pkv_pool* p, int32_t n_seqs, int32_t Hq, int32_t partition_tokens, int32_t window,
                       DecodePlan* out, bool defer = false) {
  const pkv_pool_desc& d = p->desc;
  if (n_seqs < 0 || Hq <= 0 || Hq % d.num_kv_heads != 0) return PKV_ERR_INVALID;
  if (d.block_size % pkv_dev::kChunk != 0) return PKV_ERR_INVALID;
  if (partition_tokens < 0 || partition_tokens % pkv_dev::kChunk != 0) return PKV_ERR_INVALID;
  if (n_seqs > 16384) return PKV_ERR_INVALID;
  const int g = Hq / d.num_kv_heads;
  DecodePlan pl;
  pl.k = pick_kernels(d.dtype, d.head_dim, g);
  if (!pl.k.decode) return PKV_ERR_INVALID;
  pl.nw = env_int("PKV_DECODE_WARPS", 4);
  if (pl.nw > 4) pl.nw = 4;   // the decode kernels are compiled for at most 128 threads per CTA
  pl.stages = env_int("PKV_DECODE_STAGES", 2);
  // deferred mode: bf16 pools (the only ones with a deferred instantiation), at most 4 stages (each
  // warp's stage tasks live in the CTA's scan scratch)
  pl.defer = defer && pl.k.decode_defer != nullptr && pl.stages <= 4;
  const void* kern = reinterpret_cast<const void*>(pl.defer ? pl.k.decode_defer : pl.k.decode);
  pl.smem = pkv_dev::decode_smem_bytes(pl.nw, pl.stages, pl.k.stage_bytes, n_seqs, partition_tokens > 0, window > 0);
  // every CTA keeps per-sequence prefix sums in shared memory: the batch must fit beside the ring
  const size_t smem_max = max_smem_optin();
  if (smem_max == 0) return PKV_ERR_CUDA;
  if (pl.smem > smem_max) return PKV_ERR_INVALID;
  if (!ensure_smem(kern, pl.smem)) return PKV_ERR_CUDA;
  const int per_sm = occupancy(kern, pl.nw * 32, pl.smem);
  const int sms = num_sms();
  if (per_sm <= 0 || sms <= 0) return PKV_ERR_CUDA;
  pl.grid = sms * per_sm;
  pl.warps = pl.grid * pl.nw;
  pl.n_units = static_cast<int64_t>(n_seqs) * d.num_kv_heads;
  if (partition_tokens > 0) {
    pl.part_chunks = partition_tokens / pkv_dev::kChunk;
    const int64_t max_chunks = (static_cast<int64_t>(d.max_blocks_per_seq) * d.block_size) / pkv_dev::kChunk;
    pl.max_parts = static_cast<int>((max_chunks + pl.part_chunks - 1) / pl.part_chunks);
    pl.n_slots = pl.n_units * pl.max_parts;
  } else if (pl.defer) {
    pl.max_tasks = 4 * pl.warps;   // balanced mode: slots 2 t, 2 t + 1 of task t
    pl.n_slots = 2 * static_cast<int64_t>(pl.max_tasks);
  } else {
    pl.n_slots = 2 * static_cast<int64_t>(pl.warps);
  }
  if (pl.max_parts > 0xffff || pl.warps > 0xffff) return PKV_ERR_INVALID;   // 16-bit arrival counts
  const size_t count_bytes = static_cast<size_t>(pl.n_units) * sizeof(unsigned long long);
  pl.off_ml = round_up(count_bytes, 256);
  pl.off_o = pl.off_ml + round_up(static_cast<size_t>(pl.n_slots) * g * 2 * sizeof(float), 256);
  pl.ws_bytes = pl.off_o + static_cast<size_t>(pl.n_slots) * g * d.head_dim * sizeof(float);
  // deferred mode: after the partials, [part_chunks, T1, T2, NP1 (2 words), pref[0..n], ipref[0..n]]
  // for the merge kernel
  if (pl.defer) {
    pl.off_meta = round_up(pl.ws_bytes, 256);
    pl.ws_bytes = pl.off_meta + (5 + 2 * (static_cast<size_t>(n_seqs) + 1)) * sizeof(int32_t);
  }
  *out = pl;
  return PKV_OK;
}

pkv_status decode_launch(const pkv_pool* p, float* out, const void* q, const void* k_cache, const void* v_cache,
                         const float* k_scale, const float* v_scale, const int32_t* block_tables,
                         const int32_t* context_lens, int32_t n_seqs, int32_t num_q_heads, float scale,
                         int32_t window, int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                         void* stream, int32_t start = 0, float* lse_out = nullptr,
                         bool defer = false, int32_t late_wait = 0, unsigned long long tag = 0,
                         DecodePlan* plan_out = nullptr);
pkv_status merge_launch(const pkv_pool* p, const DecodePlan& pl, unsigned char* ws, float* out, int32_t n_seqs,
                        int32_t Hq, const float* lse_s, const float* part_o, const float* part_lse, int32_t n_split,
                        const int32_t* block_tables, int32_t prefix_blocks, cudaStream_t s);

}  // namespace

extern "C" {

pkv_status pkv_reshape_and_cache(const pkv_pool* p, const void* k, const void* v, const int64_t* slots,
                                 int32_t n_tokens, void* k_cache, void* v_cache, void* stream) {
  if (!p || n_tokens < 0) return PKV_ERR_INVALID;
  if (n_tokens == 0) return PKV_OK;
  if (!k || !v || !slots || !k_cache || !v_cache) return PKV_ERR_INVALID;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(slots) & 7u))
    return PKV_ERR_INVALID;
  const pkv_pool_desc& d = p->desc;
  if (d.dtype == PKV_FP8) return PKV_ERR_INVALID;   // fp8 pools quantise: pkv_reshape_and_cache_fp8
  const int row_bytes = d.head_dim * pkv::elem_bytes(d.dtype);
  if (row_bytes % 16 != 0) return PKV_ERR_INVALID;
  const int ppr = row_bytes / 16;
  const int64_t total = static_cast<int64_t>(n_tokens) * d.num_kv_heads * ppr;
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int grid = static_cast<int>(want < 65535 * 4 ? want : 65535 * 4);
  const cudaError_t e = launch(pkv_dev::reshape_and_cache_kernel, dim3(grid), dim3(threads), 0,
                               static_cast<cudaStream_t>(stream), static_cast<const uint4*>(k),
                               static_cast<const uint4*>(v), slots, n_tokens, d.num_kv_heads, ppr, d.block_size,
                               static_cast<int64_t>(d.num_blocks) * d.block_size, static_cast<uint4*>(k_cache),
                               static_cast<uint4*>(v_cache), p->d_err_word);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_copy_blocks(const pkv_pool* p, void* const* k_caches, void* const* v_caches, const int32_t* pairs,
                           int32_t n_pairs, void* stream) {
  if (!p || n_pairs < 0) return PKV_ERR_INVALID;
  if (n_pairs == 0) return PKV_OK;
  const pkv_pool_desc& d = p->desc;
  if (d.dtype == PKV_FP8) return PKV_ERR_INVALID;   // fp8 blocks carry scales: pkv_copy_blocks_fp8
  if (!k_caches || !v_caches || !pairs || d.num_layers > pkv_dev::kMaxLayers) return PKV_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(pairs) & 7u) return PKV_ERR_INVALID;
  pkv_dev::LayerCaches lc;
  std::memset(&lc, 0, sizeof lc);
  for (int l = 0; l < d.num_layers; ++l) {
    if (!k_caches[l] || !v_caches[l] || !aligned16(k_caches[l]) || !aligned16(v_caches[l])) return PKV_ERR_INVALID;
    lc.k[l] = static_cast<uint4*>(k_caches[l]);
    lc.v[l] = static_cast<uint4*>(v_caches[l]);
  }
  const int64_t block_bytes =
      static_cast<int64_t>(d.num_kv_heads) * d.block_size * d.head_dim * pkv::elem_bytes(d.dtype);
  if (block_bytes % 16 != 0) return PKV_ERR_INVALID;
  const int64_t grid = static_cast<int64_t>(n_pairs) * d.num_layers;
  if (grid > 0x7fffffff) return PKV_ERR_INVALID;
  const cudaError_t e = launch(pkv_dev::copy_blocks_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0,
                               static_cast<cudaStream_t>(stream), lc, pairs, d.num_layers, block_bytes / 16,
                               d.num_blocks, p->d_err_word);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_paged_prefill(const pkv_pool* p, float* out, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens, const int32_t* cu_q,
                             int32_t n_seqs, int32_t total_q, int32_t num_q_heads, float scale, int32_t window,
                             void* stream) {
  if (!p || n_seqs < 0 || total_q < 0 || window < 0) return PKV_ERR_INVALID;
  if (n_seqs == 0 || total_q == 0) return PKV_OK;
  const pkv_pool_desc& d = p->desc;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !cu_q) return PKV_ERR_INVALID;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(cu_q) & 3u))
    return PKV_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return PKV_ERR_INVALID;
  if (d.dtype != PKV_BF16 || (d.head_dim != 64 && d.head_dim != 128) || d.block_size % pkv_dev::kChunk != 0)
    return PKV_ERR_INVALID;
  if (num_q_heads <= 0 || num_q_heads % d.num_kv_heads != 0) return PKV_ERR_INVALID;
  if (n_seqs > 16384 || d.max_blocks_per_seq > 8192) return PKV_ERR_INVALID;
  const int g = num_q_heads / d.num_kv_heads;
  const int64_t rows = static_cast<int64_t>(d.num_blocks) * d.num_kv_heads * d.block_size;
  if (rows > 0x7fffffffLL || d.num_kv_heads > 65535) return PKV_ERR_INVALID;
  pkv_dev::PrefillArgs a;
  std::memset(&a, 0, sizeof a);   // fields of the shared-prefix mode stay off
  a.out = out;
  a.q = q;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.cu_q = cu_q;
  a.n_seqs = n_seqs;
  a.Hq = num_q_heads;
  a.Hkv = d.num_kv_heads;
  a.B = d.block_size;
  a.NB = d.num_blocks;
  a.MB = d.max_blocks_per_seq;
  a.window = window;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err = p->d_err_word;
  a.stages = 0;   // the tcgen05 kernel fixes its ring depth at compile time
  a.total_q = total_q;
  a.shared_len = 0;
  a.split_keys = 0;
  a.part_o = nullptr;
  a.part_lse = nullptr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (prefill_path_tc() && n_seqs <= kPrefillTcMaxSeqs) return tc_prefill_launch(p, a, k_cache, v_cache, st, -1);
  using PK = void (*)(pkv_dev::PrefillArgs, pkv_dev::TmaMaps);
  PK kern = nullptr;
  int tq = 0, stage_bytes = 0, q_bytes = 0;
#define PKV_PREFILL_CASE(DD, GG)                                       \
  if (d.head_dim == DD && g == GG) {                                   \
    kern = pkv_dev::paged_prefill_kernel<DD, GG>;                      \
    tq = pkv_dev::PrefillShape<DD, GG>::TQ;                            \
    stage_bytes = pkv_dev::PrefillShape<DD, GG>::kStageBytes;          \
    q_bytes = pkv_dev::PrefillShape<DD, GG>::kQBytes;                  \
  }
  PKV_PREFILL_CASE(64, 1) PKV_PREFILL_CASE(64, 2) PKV_PREFILL_CASE(64, 3) PKV_PREFILL_CASE(64, 4)
  PKV_PREFILL_CASE(64, 5) PKV_PREFILL_CASE(64, 6) PKV_PREFILL_CASE(64, 7) PKV_PREFILL_CASE(64, 8)
  PKV_PREFILL_CASE(128, 1) PKV_PREFILL_CASE(128, 2) PKV_PREFILL_CASE(128, 3) PKV_PREFILL_CASE(128, 4)
  PKV_PREFILL_CASE(128, 5) PKV_PREFILL_CASE(128, 6) PKV_PREFILL_CASE(128, 7) PKV_PREFILL_CASE(128, 8)
#undef PKV_PREFILL_CASE
  if (!kern) return PKV_ERR_INVALID;
  const int stages = env_int("PKV_PREFILL_STAGES", 4);
  const size_t smem = pkv_dev::prefill_smem_bytes(stages, stage_bytes, q_bytes, n_seqs, d.max_blocks_per_seq);
  if (!ensure_smem(reinterpret_cast<const void*>(kern), smem)) return PKV_ERR_CUDA;
  pkv_dev::TmaMaps maps;
  std::memset(&maps, 0, sizeof maps);
  if (!encode_cache_map(&maps.k, k_cache, d) || !encode_cache_map(&maps.v, v_cache, d)) return PKV_ERR_CUDA;
  a.stages = stages;
  const int64_t tiles_ub = (static_cast<int64_t>(total_q) + tq - 1) / tq + n_seqs;   // >= sum of tiles
  if (tiles_ub > 0x7fffffffLL) return PKV_ERR_INVALID;
  if (launch(kern, dim3(static_cast<unsigned>(tiles_ub), d.num_kv_heads), dim3(128), smem, st, a, maps) !=
          cudaSuccess ||
      cudaGetLastError() != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

size_t pkv_decode_workspace_bytes(const pkv_pool* p, int32_t n_seqs, int32_t num_q_heads, int32_t partition_tokens) {
  if (!p) return 0;
  DecodePlan pl;
  if (plan_decode(p, n_seqs, num_q_heads, partition_tokens, 0, &pl, decode_defer_wanted(partition_tokens)) != PKV_OK)
    return 0;
  return pl.ws_bytes;
}

pkv_status pkv_paged_decode(const pkv_pool* p, float* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens, int32_t n_seqs,
                            int32_t num_q_heads, float scale, int32_t partition_tokens, void* workspace,
                            size_t workspace_bytes, void* stream) {
  return pkv_paged_decode_window(p, out, q, k_cache, v_cache, block_tables, context_lens, n_seqs, num_q_heads, scale,
                                 0, partition_tokens, workspace, workspace_bytes, stream);
}

pkv_status pkv_paged_decode_window(const pkv_pool* p, float* out, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                                   int32_t n_seqs, int32_t num_q_heads, float scale, int32_t window,
                                   int32_t partition_tokens, void* workspace, size_t workspace_bytes, void* stream) {
  if (p && p->desc.dtype == PKV_FP8) return PKV_ERR_INVALID;   // pkv_paged_decode_fp8
  DecodePlan pl;
  const pkv_status r =
      decode_launch(p, out, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens, n_seqs, num_q_heads,
                    scale, window, partition_tokens, workspace, workspace_bytes, stream, 0, nullptr,
                    decode_defer_wanted(partition_tokens), 0, 0, &pl);
  if (r != PKV_OK || n_seqs == 0 || !pl.defer) return r;
  return merge_launch(p, pl, static_cast<unsigned char*>(workspace), out, n_seqs, num_q_heads, nullptr, nullptr,
                      nullptr, 0, block_tables, 0, static_cast<cudaStream_t>(stream));
}

pkv_status pkv_paged_decode_fp8(const pkv_pool* p, float* out, const void* q, const void* k_cache,
                                const void* v_cache, const float* k_scale, const float* v_scale,
                                const int32_t* block_tables, const int32_t* context_lens, int32_t n_seqs,
                                int32_t num_q_heads, float scale, int32_t window, int32_t partition_tokens,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (!p || p->desc.dtype != PKV_FP8) return PKV_ERR_INVALID;
  if (n_seqs > 0 && (!k_scale || !v_scale || !aligned16(k_scale) || !aligned16(v_scale))) return PKV_ERR_INVALID;
  DecodePlan pl;
  const pkv_status r =
      decode_launch(p, out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, n_seqs, num_q_heads,
                    scale, window, partition_tokens, workspace, workspace_bytes, stream, 0, nullptr,
                    decode_defer_wanted(partition_tokens), 0, 0, &pl);
  if (r != PKV_OK || n_seqs == 0 || !pl.defer) return r;
  return merge_launch(p, pl, static_cast<unsigned char*>(workspace), out, n_seqs, num_q_heads, nullptr, nullptr,
                      nullptr, 0, block_tables, 0, static_cast<cudaStream_t>(stream));
}

pkv_status pkv_reshape_and_cache_fp8(const pkv_pool* p, const void* k, const void* v, const int64_t* slots,
                                     int32_t n_tokens, void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                                     void* stream) {
  if (!p || n_tokens < 0 || p->desc.dtype != PKV_FP8) return PKV_ERR_INVALID;
  if (n_tokens == 0) return PKV_OK;
  const pkv_pool_desc& d = p->desc;
  if (d.head_dim != 64 && d.head_dim != 128) return PKV_ERR_INVALID;
  if (!k || !v || !slots || !k_cache || !v_cache || !k_scale || !v_scale) return PKV_ERR_INVALID;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_scale) ||
      !aligned16(v_scale) || (reinterpret_cast<uintptr_t>(slots) & 7u))
    return PKV_ERR_INVALID;
  const int64_t rows = static_cast<int64_t>(n_tokens) * d.num_kv_heads;
  const int warps_per_cta = 8;
  const int64_t want = (rows + warps_per_cta - 1) / warps_per_cta;
  const int grid = static_cast<int>(want < 65535 * 4 ? want : 65535 * 4);
  auto kern = d.head_dim == 128 ? pkv_dev::reshape_and_cache_fp8_kernel<128> : pkv_dev::reshape_and_cache_fp8_kernel<64>;
  const cudaError_t e = launch(kern, dim3(grid), dim3(32 * warps_per_cta), 0, static_cast<cudaStream_t>(stream),
                               static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), slots,
                               n_tokens, d.num_kv_heads, d.block_size,
                               static_cast<int64_t>(d.num_blocks) * d.block_size, static_cast<uint8_t*>(k_cache),
                               static_cast<uint8_t*>(v_cache), k_scale, v_scale, p->d_err_word);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_copy_blocks_fp8(const pkv_pool* p, void* const* k_caches, void* const* v_caches,
                               void* const* k_scales, void* const* v_scales, const int32_t* pairs, int32_t n_pairs,
                               void* stream) {
  if (!p || n_pairs < 0 || p->desc.dtype != PKV_FP8) return PKV_ERR_INVALID;
  if (n_pairs == 0) return PKV_OK;
  const pkv_pool_desc& d = p->desc;
  if (!k_caches || !v_caches || !k_scales || !v_scales || !pairs || d.num_layers > pkv_dev::kMaxLayers)
    return PKV_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(pairs) & 7u) return PKV_ERR_INVALID;
  pkv_dev::LayerCaches codes, scales;
  std::memset(&codes, 0, sizeof codes);
  std::memset(&scales, 0, sizeof scales);
  for (int l = 0; l < d.num_layers; ++l) {
    if (!k_caches[l] || !v_caches[l] || !k_scales[l] || !v_scales[l] || !aligned16(k_caches[l]) ||
        !aligned16(v_caches[l]) || !aligned16(k_scales[l]) || !aligned16(v_scales[l]))
      return PKV_ERR_INVALID;
    codes.k[l] = static_cast<uint4*>(k_caches[l]);
    codes.v[l] = static_cast<uint4*>(v_caches[l]);
    scales.k[l] = static_cast<uint4*>(k_scales[l]);
    scales.v[l] = static_cast<uint4*>(v_scales[l]);
  }
  const int64_t code_bytes = static_cast<int64_t>(d.num_kv_heads) * d.block_size * d.head_dim;
  const int64_t scale_bytes = static_cast<int64_t>(d.num_kv_heads) * d.block_size * 4;
  if (code_bytes % 16 != 0 || scale_bytes % 16 != 0) return PKV_ERR_INVALID;
  const int64_t grid = static_cast<int64_t>(n_pairs) * d.num_layers;
  if (grid > 0x7fffffff) return PKV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch(pkv_dev::copy_blocks_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, codes, pairs,
             d.num_layers, code_bytes / 16, d.num_blocks, p->d_err_word) != cudaSuccess ||
      launch(pkv_dev::copy_blocks_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, scales, pairs,
             d.num_layers, scale_bytes / 16, d.num_blocks, p->d_err_word) != cudaSuccess ||
      cudaGetLastError() != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

}  // extern "C"

namespace {

pkv_status decode_launch(const pkv_pool* p, float* out, const void* q, const void* k_cache, const void* v_cache,
                         const float* k_scale, const float* v_scale, const int32_t* block_tables,
                         const int32_t* context_lens, int32_t n_seqs, int32_t num_q_heads, float scale,
                         int32_t window, int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                         void* stream, int32_t start, float* lse_out, bool defer_req,
                         int32_t late_wait, unsigned long long tag, DecodePlan* plan_out) {
  if (!p || window < 0) return PKV_ERR_INVALID;
  if (n_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_INVALID;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return PKV_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return PKV_ERR_INVALID;
  DecodePlan pl;
  const pkv_status st =
      plan_decode(p, n_seqs, num_q_heads, partition_tokens, (window > 0 || start > 0) ? 1 : 0, &pl, defer_req);
  const bool defer = pl.defer;
  if (st != PKV_OK) return st;
  if (workspace_bytes < pl.ws_bytes || (pl.ws_bytes > 0 && (!workspace || !aligned16(workspace))))
    return PKV_ERR_INVALID;
  const pkv_pool_desc& d = p->desc;
  DecodeArgs a;
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  a.ws_count = reinterpret_cast<unsigned long long*>(ws);
  a.ws_ml = reinterpret_cast<float*>(ws + pl.off_ml);
  a.ws_o = reinterpret_cast<float*>(ws + pl.off_o);
  a.n_seqs = n_seqs;
  a.Hq = num_q_heads;
  a.Hkv = d.num_kv_heads;
  a.B = d.block_size;
  a.NB = d.num_blocks;
  a.MB = d.max_blocks_per_seq;
  a.part_chunks = pl.part_chunks;
  a.max_parts = pl.max_parts;
  a.stages = pl.stages;
  a.total_warps = pl.warps;
  a.window = window;
  a.scale_log2 = scale * 1.4426950408889634f;
  pkv_dev::TmaMaps maps;
  std::memset(&maps, 0, sizeof maps);
  if (pl.k.maps != MAPS_NONE) {
    const int64_t rows = static_cast<int64_t>(d.num_blocks) * d.num_kv_heads * d.block_size *
                         (pl.k.maps == MAPS_FP8 ? d.head_dim / d.block_size + 1 : 1);
    if (rows > 0x7fffffffLL) return PKV_ERR_INVALID;   // tensor coordinates are 32-bit
    if (pl.k.maps == MAPS_BF16 && d.head_dim == 128) {   // MmaMath<128, G> copies through 3-D maps
      if (!encode_cache_map_halves(&maps.k, k_cache, d) || !encode_cache_map_halves(&maps.v, v_cache, d))
        return PKV_ERR_CUDA;
    } else if (pl.k.maps == MAPS_BF16) {
      if (!encode_cache_map(&maps.k, k_cache, d) || !encode_cache_map(&maps.v, v_cache, d)) return PKV_ERR_CUDA;
    } else if (!encode_fp8_maps(&maps, k_cache, v_cache, d)) {
      return PKV_ERR_CUDA;
    }
  }
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  // Balanced mode gives every warp at least 16 chunks (256 tokens), 8 when the whole call has fewer
  // than 8192 chunks: below that, cutting units into more parts costs more in merges than the extra
  // warps gain (measured on batches of 4-256 sequences of 256-4096 tokens; problems with more than
  // 16 chunks per warp are unaffected).
  a.min_chunks = env_int("PKV_DECODE_MIN_CHUNKS", 16);
  a.tag = tag != 0 ? tag : next_call_tag();
  a.err = p->d_err_word;
  a.start = start;
  a.lse_out = lse_out;
  a.defer_meta = defer ? reinterpret_cast<int32_t*>(ws + pl.off_meta) : nullptr;
  a.max_tasks = pl.max_tasks;
  // deferred mode: chunks per task (no arrivals, so cutting units costs no fences; small tasks balance)
  if (defer) a.min_chunks = env_int("PKV_CASCADE_TASK_CHUNKS", 16);
  a.late_wait = late_wait;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch(pl.defer ? pl.k.decode_defer : pl.k.decode, dim3(pl.grid), dim3(pl.nw * 32), pl.smem, s, a, maps) !=
          cudaSuccess ||
      cudaGetLastError() != cudaSuccess)
    return PKV_ERR_CUDA;
  if (plan_out) *plan_out = pl;
  return PKV_OK;
}

// The merge kernel after a deferred-mode decode (plan pl, workspace ws): the rows of units cut by
// task boundaries, and with n_split > 0 the shared-prefix splits of every row.
pkv_status merge_launch(const pkv_pool* p, const DecodePlan& pl, unsigned char* ws, float* out, int32_t n_seqs,
                        int32_t Hq, const float* lse_s, const float* part_o, const float* part_lse, int32_t n_split,
                        const int32_t* block_tables, int32_t prefix_blocks, cudaStream_t s) {
  const pkv_pool_desc& d = p->desc;
  pkv_dev::CascadeMergeArgs m;
  m.out = out;
  m.lse_s = lse_s;
  m.part_o = part_o;
  m.part_lse = part_lse;
  m.dec_o = reinterpret_cast<const float*>(ws + pl.off_o);
  m.dec_ml = reinterpret_cast<const float*>(ws + pl.off_ml);
  m.meta = reinterpret_cast<const int32_t*>(ws + pl.off_meta);
  m.max_parts = pl.max_parts;
  m.task_ctr = reinterpret_cast<unsigned long long*>(ws);   // the decode's first workspace word
  m.tables = block_tables;
  m.n_rows = static_cast<int64_t>(n_seqs) * Hq;
  m.D = d.head_dim;
  m.G = Hq / d.num_kv_heads;
  m.Hkv = d.num_kv_heads;
  m.n_split = n_split;
  m.MB = d.max_blocks_per_seq;
  m.n_seqs = n_seqs;
  m.prefix_blocks = prefix_blocks;
  m.err = p->d_err_word;
  // one wave: a warp per row, rows beyond the resident warps taken grid-stride
  const int per_sm = occupancy(reinterpret_cast<const void*>(pkv_dev::merge_prefix_kernel), 256, 0);
  const int64_t wave = static_cast<int64_t>(per_sm > 0 ? per_sm : 1) * num_sms();
  const int64_t want = (m.n_rows + 7) / 8;
  const int64_t blocks = want < wave ? want : wave;
  if (launch(pkv_dev::merge_prefix_kernel, dim3(static_cast<unsigned>(blocks > 0 ? blocks : 1)), dim3(256), 0, s,
             m) != cudaSuccess ||
      cudaGetLastError() != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

}  // namespace

namespace {

// Shared-prefix decode: workspace layout and key splits.
struct SharedPlan {
  DecodePlan dec;
  int32_t shared_len = 0, split_keys = 0, n_split = 0, item_tokens = 0;
  int64_t grid_items = 0;
  size_t off_lse = 0, off_plse = 0, off_po = 0, bytes = 0;
};

pkv_status plan_shared(const pkv_pool* p, int32_t n_seqs, int32_t Hq, int32_t prefix_blocks, SharedPlan* out) {
  const pkv_pool_desc& d = p->desc;
  if (d.dtype != PKV_BF16 || (d.head_dim != 64 && d.head_dim != 128) || d.block_size % pkv_dev::kChunk != 0)
    return PKV_ERR_INVALID;
  if (n_seqs <= 0 || Hq <= 0 || Hq % d.num_kv_heads != 0) return PKV_ERR_INVALID;
  if (prefix_blocks <= 0 || prefix_blocks > d.max_blocks_per_seq) return PKV_ERR_INVALID;
  const int g = Hq / d.num_kv_heads;
  SharedPlan sp;
  sp.item_tokens = tc_item_tokens(d.head_dim, g);
  if (sp.item_tokens == 0) return PKV_ERR_INVALID;
  const pkv_status st = plan_decode(p, n_seqs, Hq, 0, 1, &sp.dec, true);
  if (st != PKV_OK) return st;
  sp.shared_len = prefix_blocks * d.block_size;
  // key splits of the shared prefix: work items for about a quarter of the SMs. The tensor-core
  // kernel runs beside the suffix decode, and each SM it holds is one the decode cannot stream on
  // (its copies in flight are bounded by shared memory per SM); longer key ranges per item cost
  // less than that (measured on 128 children of a 1,024-token prompt: 2 splits of 512 keys, 32 CTAs,
  // against 8 splits of 128 keys, 128 CTAs).
  const int64_t items_per_split = (static_cast<int64_t>(n_seqs) + sp.item_tokens - 1) / sp.item_tokens * d.num_kv_heads;
  const int sms = num_sms();
  if (sms <= 0) return PKV_ERR_CUDA;
  int64_t ns = (sms / 4 + items_per_split / 2) / items_per_split;
  const int64_t max_split = (sp.shared_len + 63) / 64;
  ns = ns < 1 ? 1 : (ns > max_split ? max_split : ns);
  sp.split_keys = static_cast<int32_t>(((sp.shared_len + ns - 1) / ns + 63) / 64 * 64);
  const int forced = env_int("PKV_SHARED_SPLIT_KEYS", 0);   // tuning: keys per split (multiple of 64)
  if (forced >= 64 && forced % 64 == 0) sp.split_keys = forced;
  sp.n_split = (sp.shared_len + sp.split_keys - 1) / sp.split_keys;
  sp.grid_items = items_per_split * sp.n_split;
  const size_t rows = static_cast<size_t>(n_seqs) * Hq;
  if (!sp.dec.defer) return PKV_ERR_INVALID;
  sp.off_lse = round_up(sp.dec.ws_bytes, 256);
  sp.off_plse = sp.off_lse + round_up(rows * sizeof(float), 256);
  sp.off_po = sp.off_plse + round_up(static_cast<size_t>(sp.n_split) * rows * sizeof(float), 256);
  sp.bytes = sp.off_po + static_cast<size_t>(sp.n_split) * rows * d.head_dim * sizeof(float);
  *out = sp;
  return PKV_OK;
}

}  // namespace

extern "C" {

size_t pkv_decode_shared_prefix_workspace_bytes(const pkv_pool* p, int32_t n_seqs, int32_t num_q_heads,
                                                int32_t prefix_blocks) {
  if (!p) return 0;
  if (prefix_blocks == 0) return pkv_decode_workspace_bytes(p, n_seqs, num_q_heads, 0);
  SharedPlan sp;
  if (plan_shared(p, n_seqs, num_q_heads, prefix_blocks, &sp) != PKV_OK) return 0;
  return sp.bytes;
}

pkv_status pkv_paged_decode_shared_prefix(const pkv_pool* p, float* out, const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          const int32_t* context_lens, int32_t n_seqs, int32_t num_q_heads,
                                          float scale, int32_t prefix_blocks, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  if (!p || n_seqs < 0 || prefix_blocks < 0) return PKV_ERR_INVALID;
  if (n_seqs == 0) return PKV_OK;
  if (prefix_blocks == 0)
    return pkv_paged_decode(p, out, q, k_cache, v_cache, block_tables, context_lens, n_seqs, num_q_heads, scale, 0,
                            workspace, workspace_bytes, stream);
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace) return PKV_ERR_INVALID;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return PKV_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return PKV_ERR_INVALID;
  SharedPlan sp;
  const pkv_status st = plan_shared(p, n_seqs, num_q_heads, prefix_blocks, &sp);
  if (st != PKV_OK) return st;
  if (workspace_bytes < sp.bytes) return PKV_ERR_INVALID;
  const pkv_pool_desc& d = p->desc;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  float* lse_s = reinterpret_cast<float*>(ws + sp.off_lse);
  float* part_lse = reinterpret_cast<float*>(ws + sp.off_plse);
  float* part_o = reinterpret_cast<float*>(ws + sp.off_po);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // 1. the shared prefix once for every row (tensor-core kernel, key splits); once past its own
  // dependency wait it lets the decode launch (decode CTAs take the SMs it leaves free and, by dynamic
  // tasks, the rest as its CTAs finish), and it installs the decode's call tag in the task counter.
  pkv_dev::PrefillArgs a;
  std::memset(&a, 0, sizeof a);
  a.out = nullptr;
  a.q = q;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.cu_q = nullptr;
  a.n_seqs = 1;
  a.Hq = num_q_heads;
  a.Hkv = d.num_kv_heads;
  a.B = d.block_size;
  a.NB = d.num_blocks;
  a.MB = d.max_blocks_per_seq;
  a.window = 0;
  a.stages = 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err = p->d_err_word;
  a.total_q = n_seqs;
  a.shared_len = sp.shared_len;
  a.split_keys = sp.split_keys;
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.early_trigger = 1;
  const unsigned long long tag = next_call_tag();   // the decode's call tag
  a.task_ctr = reinterpret_cast<unsigned long long*>(ws);
  a.task_tag = tag;
  pkv_status r = tc_prefill_launch(p, a, k_cache, v_cache, s, sp.grid_items);
  if (r != PKV_OK) return r;
  // 2. private suffixes: decode over positions [shared_len, len) with each row's log-sum-exp, in
  // deferred-merge mode (dynamic tasks; units cut by task boundaries leave partials for step 3). It
  // reads nothing step 1 writes and waits for step 1 only before completing, so that step 3 (which
  // waits for it) sees both.
  r = decode_launch(p, out, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens, n_seqs, num_q_heads,
                    scale, 0, 0, workspace, sp.dec.ws_bytes, stream, sp.shared_len, lse_s, true, 1, tag);
  if (r != PKV_OK) return r;
  // 3. log-sum-exp merge of every row's parts: suffix (final row or cut-unit partials) and prefix splits
  return merge_launch(p, sp.dec, ws, out, n_seqs, num_q_heads, lse_s, part_o, part_lse, sp.n_split, block_tables,
                      prefix_blocks, s);
}

}  // extern "C"

extern "C" {

pkv_status pkv_selftest_wait_timeout(int32_t* gave_up, void* stream) {
  pkv_dev::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(gave_up);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

static pkv_status error_status(unsigned int bits) {
  if (bits & pkv_dev::ERRBIT_TIMEOUT) return PKV_ERR_DEVICE_TIMEOUT;
  if (bits & pkv_dev::ERRBIT_BOUNDS) return PKV_ERR_DEVICE_BOUNDS;
  return PKV_OK;
}

pkv_status pkv_last_error(const pkv_pool* p) {
  if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
  unsigned int bits = 0;
  if (cudaMemcpyFromSymbol(&bits, pkv_dev::g_error_bits, sizeof bits) != cudaSuccess) return PKV_ERR_CUDA;
  const unsigned int zero = 0;
  if (bits && cudaMemcpyToSymbol(pkv_dev::g_error_bits, &zero, sizeof zero) != cudaSuccess) return PKV_ERR_CUDA;
  if (p && p->d_err_word) {   // the pool's own word as well
    unsigned int pb = 0;
    if (cudaMemcpy(&pb, p->d_err_word, sizeof pb, cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_CUDA;
    if (pb && cudaMemset(p->d_err_word, 0, sizeof pb) != cudaSuccess) return PKV_ERR_CUDA;
    bits |= pb;
  }
  return error_status(bits);
}

pkv_status pkv_pool_set_error_word(pkv_pool* p, uint32_t* d_word) {
  if (!p) return PKV_ERR_INVALID;
  if (d_word && (reinterpret_cast<uintptr_t>(d_word) & 3u)) return PKV_ERR_INVALID;
  p->d_err_word = reinterpret_cast<unsigned int*>(d_word);
  return PKV_OK;
}

pkv_status pkv_stream_error(const pkv_pool* p, void* stream) {
  if (!p || !p->d_err_word) return PKV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int bits = 0;
  // on the stream: read the word, then clear it; only this stream is waited for
  if (cudaMemcpyAsync(&bits, p->d_err_word, sizeof bits, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(p->d_err_word, 0, sizeof bits, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return PKV_ERR_CUDA;
  return error_status(bits);
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// pkv_paged_decode_static: the same decode with scratch compiled into the library, for callers
// that may not allocate device memory. The array below is part of the module image: each device
// that loads the library holds it until the process exits. Host code must not use its name as an
// address (on the host it is only a stand-in); the device address is looked up once per device
// and context (again after the device's context was reset and re-created).
// ---------------------------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

namespace {

std::mutex g_static_mu;
struct StaticScratch {
  unsigned long long ctx_id = 0;  // context the address belongs to (0: not looked up yet)
  void* ptr = nullptr;
};
StaticScratch g_static[64];

// Unique id of the calling thread's current CUDA context (cuCtxGetId: ids are never reused within
// a process, unlike context handles), or 0 if it cannot be read.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_static_scratch on the current device. It is looked up with the device
// current the first time the device is used, and again whenever the device's context is not the
// one the address was taken in (the primary context was reset and re-created), since the module
// and its array are then loaded anew.
pkv_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  unsigned long long ctx = current_context_id();   // 0 when no context is current on this thread yet
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static[dev].ptr == nullptr || ctx == 0 || g_static[dev].ctx_id != ctx) {
    void* ptr = nullptr;   // the lookup also makes the device's primary context current
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) return PKV_ERR_CUDA;
    ctx = current_context_id();
    if (ctx == 0) return PKV_ERR_CUDA;
    g_static[dev].ptr = ptr;
    g_static[dev].ctx_id = ctx;
  }
  *out = g_static[dev].ptr;
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_static(const pkv_pool* p, float* out, const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_tables,
                                              const int32_t* context_lens, int32_t n_seqs, int32_t num_q_heads,
                                              float scale, int32_t partition_tokens, void* stream) {
  if (!p) return PKV_ERR_INVALID;
  if (n_seqs == 0) return PKV_OK;
  const size_t need = pkv_decode_workspace_bytes(p, n_seqs, num_q_heads, partition_tokens);
  if (need == 0) return PKV_ERR_INVALID;
  if (need > PKV_STATIC_SCRATCH_BYTES) return PKV_ERR_SCRATCH_TOO_SMALL;
  void* scratch = nullptr;
  const pkv_status st = static_scratch(&scratch);
  if (st != PKV_OK) return st;
  return pkv_paged_decode(p, out, q, k_cache, v_cache, block_tables, context_lens, n_seqs, num_q_heads, scale,
                          partition_tokens, scratch, PKV_STATIC_SCRATCH_BYTES, stream);
}
