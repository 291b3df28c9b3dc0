// Host side of the C ABI declared in include/fattn.h: argument validation,
// tensor-map encoding, launch planning, the device status block.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fattn.h"
#include "fattn_decode_launch.h"
#include "fattn_launch.cuh"
#include "fattn_status.h"

namespace fattn {
namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 1000000000ull;  // 1 s per wait

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                   void*, const cuuint64_t*, const cuuint64_t*,
                                   const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
using AddressRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);
using CtxGetCurrentFn = CUresult (*)(CUcontext*);

struct DriverFns {
  EncodeTiledFn encode = nullptr;
  AddressRangeFn range = nullptr;
  CtxGetCurrentFn ctx_current = nullptr;
};

// Driver entry points through the runtime, so the library loads (and its
// host-side checks run) on machines without a driver.
const DriverFns& driver() {
  static const DriverFns fns = [] {
    DriverFns f;
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.encode = reinterpret_cast<EncodeTiledFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.range = reinterpret_cast<AddressRangeFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.ctx_current = reinterpret_cast<CtxGetCurrentFn>(p);
    cudaGetLastError();
    return f;
  }();
  return fns;
}

// Counter pairs for the causal kernels' run-time unit assignment: each
// launch takes the next pair (round robin) and its last CTA returns both
// words to 0.  Launches that run at the same time (other streams or host
// threads) get different pairs as long as fewer than kSchedSlots of them
// are in flight at once.  Launches enqueued into a stream capture take their
// pairs from a second ring of kSchedSlots: a captured launch keeps its pair
// for every replay of the graph (replays of one graph never overlap), and
// no ordinary launch can be handed the same pair.
constexpr int kSchedSlots = 256;

struct DeviceState {
  bool init = false;
  bool supported = false;
  int sms = 0;
  int* status = nullptr;  // kStatusWords ints, device memory
  int* sched = nullptr;   // 2 * kSchedSlots pairs of ints, device memory, zeroed once
  std::atomic<unsigned> sched_next{0};        // ordinary launches: pairs [0, kSchedSlots)
  std::atomic<unsigned> sched_next_graph{0};  // captured launches: the next kSchedSlots
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

unsigned long long wait_timeout_ns() {
  static const unsigned long long t = [] {
    const char* s = std::getenv("FATTN_WAIT_TIMEOUT_MS");
    if (s && *s) {
      const long long ms = std::atoll(s);
      if (ms > 0 && ms < 600000) return (unsigned long long)ms * 1000000ull;
    }
    return kDefaultTimeoutNs;
  }();
  return t;
}

// Make sure the calling thread has a current context.  The driver calls of
// the buffer checks (cuMemGetAddressRange) need one, and a host thread that
// has made no context-creating runtime call yet has none: there the current
// device's primary context is bound to the thread (cudaSetDevice on the
// device the thread already has, which changes nothing else).
int bind_context(int dev) {
  const DriverFns& f = driver();
  CUcontext ctx = nullptr;
  if (f.ctx_current && f.ctx_current(&ctx) == CUDA_SUCCESS && ctx) return kOk;
  if (cudaSetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return kErrCuda;
  }
  return kOk;
}

// The current device's state, created on first use (device query, status
// block allocation).  Must not first run inside a stream capture.
int current_device(DeviceState** out, int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return kErrUnsupported;
  }
  if (dev < 0 || dev >= kMaxDevices) return kErrUnsupported;
  if (const int rc = bind_context(dev); rc != kOk) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return kErrCuda;
    }
    d.sms = sms;
    d.supported = (major == 10 && minor == 3);
    if (d.supported) {
      if (cudaMalloc(&d.status, sizeof(int) * kStatusWords) != cudaSuccess ||
          cudaMemset(d.status, 0, sizeof(int) * kStatusWords) != cudaSuccess ||
          cudaMalloc(&d.sched, sizeof(int) * 4 * kSchedSlots) != cudaSuccess ||
          cudaMemset(d.sched, 0, sizeof(int) * 4 * kSchedSlots) != cudaSuccess ||
          cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        if (d.status) cudaFree(d.status);
        if (d.sched) cudaFree(d.sched);
        d.status = nullptr;
        d.sched = nullptr;
        return kErrCuda;
      }
    }
    d.init = true;
  }
  if (!d.supported) return kErrUnsupported;
  *out = &d;
  if (dev_out) *dev_out = dev;
  return kOk;
}

// Heads per group of the causal order: as many as keep the group's K and V
// (bytes_per_row per key row of one of them) within group_mib MiB of L2, so
// that the heads of the groups in flight at a group change fit with room for
// the query, output and other traffic.
// Heads per group of the causal order: as many as keep the group's K and V
// (bytes_per_row per key row of one of them) within about a quarter of L2,
// so that the heads of the two groups in flight at a group change fit with
// room for the query, output and other traffic.  The groups are made
// near-equal: each group restarts the longest-first order, so a small last
// group hands its longest units out last, when most CTAs are nearly done.
// With min_units > 0 (units of a group, n_units per head), groups are also
// merged while one would hold fewer than min_units units, since a group
// change is a restart of the order that only enough units after it can even
// out.  Measured at D = 128 (B2 H16 S4097 bf16 causal, K and V just over
// 64 MiB): groups of 15, 15 and 2 heads 944 TF, 11, 11 and 10 1117-1120,
// 16 and 16 1219-1222; B3 H11 S4096 in 16, 16 and 1 heads 917-921, in 11, 11
// and 11 1082, in 17 and 16 1189-1214.
int causal_group_heads(int BH, int S, int bytes_per_row, int n_units, int min_units) {
  const double per_head = 2.0 * (double)S * bytes_per_row;  // K and V of one head
  int g = (int)(32.0 * 1024 * 1024 / per_head);
  if (g < 1) g = 1;
  if (g >= BH) return BH;
  int groups = (BH + g - 1) / g;
  while (groups > 1 && (long long)((BH + groups - 1) / groups) * n_units < min_units) --groups;
  return (BH + groups - 1) / groups;
}

// The causal order of a launch: heads per group and whether units are handed
// out at run time.  The CTA pairs (D = 256) always take them at run time, in
// 32 MiB groups; D = 128 (16-bit, or E4M3 with elem_bytes 1) only when the
// heads form more than one group, each holding at least 1.5 units per SM;
// otherwise, and at D = 64, every head is in one group and each CTA takes
// the static snake.
void causal_order(int BH, int S, int D, int elem_bytes, int units_per_head, int sms,
                  int* group_heads, bool* run_time) {
  const int g = causal_group_heads(BH, S, D * elem_bytes, units_per_head,
                                   D == 128 ? 3 * sms / 2 : 0);
  *run_time = D == 256 || (D == 128 && g < BH);
  *group_heads = *run_time ? g : BH;
}

int* sched_pair(DeviceState* ds, cudaStream_t stream) {
  // The legacy default stream is never captured itself (and querying it
  // while another stream captures in global mode is an error), so only
  // other streams are asked.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (stream != nullptr && cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    cs = cudaStreamCaptureStatusNone;
  }
  const bool captured = cs == cudaStreamCaptureStatusActive;
  std::atomic<unsigned>& next = captured ? ds->sched_next_graph : ds->sched_next;
  const unsigned slot = next.fetch_add(1, std::memory_order_relaxed) % kSchedSlots +
                        (captured ? kSchedSlots : 0);
  return ds->sched + 2 * slot;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a);
  const uintptr_t y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// The buffer must be device (or managed) memory of the current device, and
// its allocation must hold ``bytes`` from ``p``.
int check_device_buffer(const void* p, size_t bytes, int dev) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return kErrInvalidArg;
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return kErrInvalidArg;
  if (attr.type == cudaMemoryTypeDevice && attr.device != dev) return kErrInvalidArg;
  const DriverFns& f = driver();
  if (!f.range) return kErrCuda;
  CUdeviceptr base = 0;
  size_t size = 0;
  if (f.range(&base, &size, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS)
    return kErrInvalidArg;
  if (reinterpret_cast<uintptr_t>(p) + bytes > (uintptr_t)base + size)
    return kErrInvalidArg;
  return kOk;
}

// The same for E4M3 inputs: one box is 128 columns (128 bytes) x 128 rows.
int encode_bhsd_e4m3(CUtensorMap* tm, const void* ptr, int S, int BH, int D) {
  const DriverFns& f = driver();
  if (!f.encode) return kErrCuda;
  cuuint64_t gdim[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
  cuuint64_t gstride[2] = {(cuuint64_t)D, (cuuint64_t)S * (cuuint64_t)D};
  cuuint32_t box[3] = {128, (cuuint32_t)kBM, 1};
  cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = f.encode(
      tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), gdim, gstride, box,
      estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? kOk : kErrCuda;
}

int encode_bhsd(CUtensorMap* tm, const void* ptr, int S, int BH, int D,
                bool bf16, int box_rows = kBM) {
  const DriverFns& f = driver();
  if (!f.encode) return kErrCuda;
  // [BH, S, D] viewed as 3-D (D innermost); one box is 64 columns (128 bytes,
  // the swizzle span) x box_rows rows of one head.  Rows past S read as zeros.
  cuuint64_t gdim[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
  cuuint64_t gstride[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * (cuuint64_t)D * 2};
  cuuint32_t box[3] = {(cuuint32_t)kSwizzleChunkCols, (cuuint32_t)box_rows, 1};
  cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = f.encode(
      tm, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
      3, const_cast<void*>(ptr), gdim, gstride, box, estride,
      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? kOk : kErrCuda;
}

// The K or V cache [BH, Sk, D] for the split decode kernel: boxes of 64
// columns x 32 rows (one key per lane), 128-byte swizzle.
int encode_cache(CUtensorMap* tm, const void* ptr, int Sk, int BH, int D,
                 bool bf16) {
  const DriverFns& f = driver();
  if (!f.encode) return kErrCuda;
  cuuint64_t gdim[3] = {(cuuint64_t)D, (cuuint64_t)Sk, (cuuint64_t)BH};
  cuuint64_t gstride[2] = {(cuuint64_t)D * 2, (cuuint64_t)Sk * (cuuint64_t)D * 2};
  cuuint32_t box[3] = {(cuuint32_t)decode::kBoxCols, (cuuint32_t)decode::kTileKeys, 1};
  cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = f.encode(
      tm, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
      3, const_cast<void*>(ptr), gdim, gstride, box, estride,
      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? kOk : kErrCuda;
}

struct KvPlan {
  int grid, warps, threads, smem, split_warps;
  unsigned long long records, ws_bytes;
};

// Sizes-only checks and the launch shape of the cache-attention kernels on a
// device with ``sms`` SMs: one split CTA per SM, fewer when the caches hold
// fewer tiles than the CTAs have warps.
int kvcache_checks(int B, int H, int Sq, int Sk, int D, int sms, KvPlan* plan) {
  if (B < 1 || H < 1 || Sq < 1 || Sk < 1) return kErrInvalidArg;
  if (D != 64 && D != 128) return kErrUnsupported;
  if (Sq > decode::kMaxSq) return kErrUnsupported;
  const long long bh = (long long)B * H;
  if (bh * Sq > INT_MAX || bh * Sk > INT_MAX) return kErrTooLarge;
  plan->warps = decode::warps_per_cta(D, Sq);
  plan->threads = plan->warps * 32;
  plan->smem = decode::smem_bytes(D, Sq);
  const long long max_tiles = bh * ((Sk + decode::kTileKeys - 1) / decode::kTileKeys);
  long long grid = (max_tiles + plan->warps - 1) / plan->warps;
  if (grid > sms) grid = sms;
  if (grid < 1) grid = 1;
  plan->grid = (int)grid;
  plan->split_warps = plan->grid * plan->warps;
  plan->records = (unsigned long long)plan->split_warps + (unsigned long long)bh;
  plan->ws_bytes = plan->records * (unsigned long long)Sq * (unsigned long long)(D + 1) * 4ull;
  return kOk;
}

struct Plan {
  int qt, ns, threads, smem, units_per_head, total_units;
};

// Head dims served by the CTA-pair kernel.  (At 128 the one-SM kernel with
// two query tiles per CTA is faster: 1.5 PF against 0.86 PF measured.)
bool use_pair(int D) { return D == 256; }

int host_checks(int B, int H, int S, int D, Plan* plan) {
  if (B < 1 || H < 1 || S < 1) return kErrInvalidArg;
  if (D != 64 && D != 128 && D != 256) return kErrUnsupported;
  const long long rows = (long long)B * H * S;
  if (rows > INT_MAX) return kErrTooLarge;
  if (use_pair(D)) {
    // the CTA-pair kernel: a unit is 256 query rows, one 128-row tile per SM
    plan->qt = 2;
    plan->ns = PairConfig<256>::NS;
    plan->threads = pair::PairWarps::kThreads;
    plan->smem = PairShape<256>::kSmem;
  } else if (D == 64) {
    plan->qt = FwdConfig<64>::QT;
    plan->ns = FwdConfig<64>::NS;
    plan->threads = FwdShape<64>::kThreads;
    plan->smem = FwdShape<64>::kSmem;
  } else {
    plan->qt = FwdConfig<128>::QT;
    plan->ns = FwdConfig<128>::NS;
    plan->threads = FwdShape<128>::kThreads;
    plan->smem = FwdShape<128>::kSmem;
  }
  const int rows_per_unit = kBM * plan->qt;
  plan->units_per_head = (S + rows_per_unit - 1) / rows_per_unit;
  const long long total = (long long)B * H * plan->units_per_head;
  if (total > INT_MAX) return kErrTooLarge;
  plan->total_units = (int)total;
  return kOk;
}

// ---- the allocation-free cache entry: scratch and status in static device
// arrays, device state kept without the status-block allocation

__device__ __align__(256) static unsigned char g_noalloc_scratch[FATTN_NOALLOC_SCRATCH_BYTES];
__device__ __align__(16) static int g_noalloc_status[kStatusWords];

struct NoAllocState {
  bool init = false;
  bool supported = false;
  int sms = 0;
  void* scratch = nullptr;  // device address of g_noalloc_scratch
  int* status = nullptr;    // device address of g_noalloc_status
};

NoAllocState g_noalloc[kMaxDevices];

// The current device's no-alloc state, set up on its first use: attribute
// queries and the symbols' device addresses (no allocation).
int noalloc_device(NoAllocState** out, int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return kErrUnsupported;
  }
  if (dev < 0 || dev >= kMaxDevices) return kErrUnsupported;
  if (const int rc = bind_context(dev); rc != kOk) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  NoAllocState& d = g_noalloc[dev];
  if (!d.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return kErrCuda;
    }
    d.sms = sms;
    d.supported = (major == 10 && minor == 3);
    if (d.supported) {
      void* scratch = nullptr;
      void* status = nullptr;
      if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess ||
          cudaGetSymbolAddress(&status, g_noalloc_status) != cudaSuccess) {
        cudaGetLastError();
        return kErrCuda;
      }
      d.scratch = scratch;
      d.status = static_cast<int*>(status);
    }
    d.init = true;
  }
  if (!d.supported) return kErrUnsupported;
  *out = &d;
  if (dev_out) *dev_out = dev;
  return kOk;
}

// CTAs of the persistent grid: one per SM, but for the CTA-pair kernel (D =
// 256) twice the clusters that fit at once (occupancy query, cached per
// device and mask/dtype under the library mutex).
int fwd_grid(const Plan& plan, int D, bool causal, bool bf16, int sms) {
  if (!use_pair(D)) return plan.total_units < sms ? plan.total_units : sms;
  static int fit[kMaxDevices][4] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (dev < 0 || dev >= kMaxDevices) return 0;
  int clusters = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int& slot = fit[dev][(causal ? 2 : 0) + (bf16 ? 1 : 0)];
    if (slot <= 0) slot = pair_clusters_d256(causal, bf16);
    clusters = slot;
  }
  if (clusters <= 0) return 0;
  if (plan.total_units < clusters) clusters = plan.total_units;
  return 2 * clusters;
}

// One warp waits on a shared-memory barrier that nothing completes, with the
// bounded wait every kernel of the library uses: it must give up after
// timeout_ns, record a pipeline timeout in the status block and return.
__global__ void wait_check_kernel(int* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t barrier_word;
  __shared__ int abort_flag;
  const uint32_t b = ptx::smem_u32(&barrier_word);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncwarp();
  const bool done = ptx::mbar_wait(b, 0, &abort_flag, timeout_ns);
  if (!__any_sync(0xffffffffu, done) && threadIdx.x == 0 && atomicCAS(status, 0, kErrPipelineTimeout) == 0) {
    status[1] = kRoleWaitCheck << 8;
    status[2] = (int)blockIdx.x;
  }
}

}  // namespace
}  // namespace fattn

using namespace fattn;

extern "C" {

FATTN_API int fattn_version(void) { return 100; }

FATTN_API const char* fattn_error_string(int status) {
  switch (status) {
    case FATTN_OK: return "ok";
    case FATTN_ERR_INVALID_ARG: return "invalid argument";
    case FATTN_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case FATTN_ERR_MISALIGNED: return "misaligned pointer";
    case FATTN_ERR_TOO_LARGE: return "problem too large";
    case FATTN_ERR_LAUNCH: return "kernel launch failed";
    case FATTN_ERR_PIPELINE_TIMEOUT: return "device pipeline wait timed out";
    case FATTN_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

FATTN_API int fattn_plan(int B, int H, int S, int D, int causal, int* grid,
                         int* block, int* smem_bytes, int* units,
                         int* q_tiles_per_unit, int* kv_stages) {
  Plan plan;
  const int rc = host_checks(B, H, S, D, &plan);
  if (rc != kOk) return rc;
  int g = use_pair(D) ? 2 * plan.total_units : plan.total_units;
  DeviceState* ds = nullptr;
  if (current_device(&ds, nullptr) == kOk) {
    const int fg = fwd_grid(plan, D, causal != 0, true, ds->sms);
    if (fg > 0) g = fg;
  }
  if (grid) *grid = g;
  if (block) *block = plan.threads;
  if (smem_bytes) *smem_bytes = plan.smem;
  if (units) *units = plan.total_units;
  if (q_tiles_per_unit) *q_tiles_per_unit = plan.qt;
  if (kv_stages) *kv_stages = plan.ns;
  return kOk;
}

FATTN_API int fattn_causal_order(int B, int H, int S, int D, int elem_bytes, int sms,
                                 int* group_heads, int* run_time) {
  if (sms < 1 || (elem_bytes != 1 && elem_bytes != 2)) return kErrInvalidArg;
  if (elem_bytes == 1 && D != 128) return kErrUnsupported;
  Plan plan;
  const int rc = host_checks(B, H, S, D, &plan);
  if (rc != kOk) return rc;
  int g = B * H;
  bool rt = false;
  causal_order(B * H, S, D, elem_bytes, plan.units_per_head, sms, &g, &rt);
  if (group_heads) *group_heads = g;
  if (run_time) *run_time = rt ? 1 : 0;
  return kOk;
}

FATTN_API int fattn_fwd(const void* q, const void* k, const void* v, void* o,
                        float* lse, int B, int H, int S, int D, int causal,
                        float scale, int dtype, fattn_stream_t stream) {
  // ---- host-side checks, nothing enqueued yet
  if (!q || !k || !v || !o || !lse) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  Plan plan;
  int rc = host_checks(B, H, S, D, &plan);
  if (rc != kOk) return rc;
  if (dtype != FATTN_FP16 && dtype != FATTN_BF16) return FATTN_ERR_UNSUPPORTED;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if ((a16 & 15u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return FATTN_ERR_MISALIGNED;
  const size_t rows = (size_t)B * H * S;
  const size_t tbytes = rows * (size_t)D * 2;
  const size_t lbytes = rows * sizeof(float);
  if (overlaps(o, tbytes, q, tbytes) || overlaps(o, tbytes, k, tbytes) ||
      overlaps(o, tbytes, v, tbytes) || overlaps(lse, lbytes, q, tbytes) ||
      overlaps(lse, lbytes, k, tbytes) || overlaps(lse, lbytes, v, tbytes) ||
      overlaps(lse, lbytes, o, tbytes))
    return FATTN_ERR_INVALID_ARG;

  // ---- device checks
  DeviceState* ds = nullptr;
  int dev = 0;
  rc = current_device(&ds, &dev);
  if (rc != kOk) return rc;
  if ((rc = check_device_buffer(q, tbytes, dev)) != kOk) return rc;
  if ((rc = check_device_buffer(k, tbytes, dev)) != kOk) return rc;
  if ((rc = check_device_buffer(v, tbytes, dev)) != kOk) return rc;
  if ((rc = check_device_buffer(o, tbytes, dev)) != kOk) return rc;
  if ((rc = check_device_buffer(lse, lbytes, dev)) != kOk) return rc;

  const bool bf16 = dtype == FATTN_BF16;
  const int BH = B * H;
  CUtensorMap tm_q, tm_k, tm_v;
  // the CTA-pair kernel loads K in halves of 64 keys
  if (encode_bhsd(&tm_q, q, S, BH, D, bf16) != kOk ||
      encode_bhsd(&tm_k, k, S, BH, D, bf16, use_pair(D) ? 64 : kBM) != kOk ||
      encode_bhsd(&tm_v, v, S, BH, D, bf16) != kOk)
    return FATTN_ERR_CUDA;

  LaunchArgs a;
  a.tm_q = &tm_q;
  a.tm_k = &tm_k;
  a.tm_v = &tm_v;
  a.params.o = o;
  a.params.lse = lse;
  a.params.status = ds->status;
  a.params.S = S;
  a.params.BH = BH;
  a.params.n_kv_tiles = (S + kBN - 1) / kBN;
  a.params.n_units = plan.units_per_head;
  a.params.total_units = plan.total_units;
  a.params.scale_log2 = (float)((double)scale * 1.4426950408889634);
  a.params.o_scale = 1.0f;
  a.params.timeout_ns = wait_timeout_ns();
  a.grid = fwd_grid(plan, D, causal != 0, bf16, ds->sms);
  if (a.grid <= 0) return FATTN_ERR_LAUNCH;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  // Causal kernels at D = 256 hand units out at run time over head groups
  // and need a counter; so do those at D = 128 when the K and V of all heads
  // exceed one group.  Otherwise (and at D = 64) each CTA takes the static
  // snake over the longest-first order of every head: with K and V resident
  // in L2 the order costs no DRAM traffic, and the static order measured
  // faster (B1 H32 S2048 D128 fp16 causal: 926-934 against 879 TF).  At
  // D = 128 groups hold at least 1.5 units per CTA; on the CTA pairs merging
  // measured no gain (B2 H16 S4097 D256: 1041 against 1110 TF in two groups
  // of 16 rather than 32 MiB ones).
  int group = BH;
  bool run_time_units = false;
  if (causal) causal_order(BH, S, D, 2, plan.units_per_head, ds->sms, &group, &run_time_units);
  a.params.sched = run_time_units ? sched_pair(ds, a.stream) : nullptr;
  a.params.group_heads = group;

  const cudaError_t e = D == 64    ? launch_fwd_d64(causal != 0, bf16, a)
                        : D == 128 ? launch_fwd_d128(causal != 0, bf16, a)
                                   : launch_fwd_d256(causal != 0, bf16, a);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FATTN_ERR_LAUNCH;
  }
  return FATTN_OK;
}

FATTN_API int fattn_kvcache_plan(int B, int H, int Sq, int Sk, int D,
                                 unsigned long long* workspace_bytes, int* grid,
                                 int* block, int* smem_bytes, int* split_warps) {
  DeviceState* ds = nullptr;
  int rc = current_device(&ds, nullptr);
  if (rc != kOk) return rc;
  KvPlan plan;
  rc = kvcache_checks(B, H, Sq, Sk, D, ds->sms, &plan);
  if (rc != kOk) return rc;
  if (workspace_bytes) *workspace_bytes = plan.ws_bytes;
  if (grid) *grid = plan.grid;
  if (block) *block = plan.threads;
  if (smem_bytes) *smem_bytes = plan.smem;
  if (split_warps) *split_warps = plan.split_warps;
  return kOk;
}

FATTN_API int fattn_fwd_kvcache(const void* q, const void* k_cache,
                                const void* v_cache, const int* cache_lens,
                                void* o, float* lse, int B, int H, int Sq,
                                int Sk, int D, int causal, float scale,
                                int dtype, void* workspace,
                                unsigned long long workspace_bytes,
                                fattn_stream_t stream) {
  // ---- host-side checks, nothing enqueued yet
  if (!q || !k_cache || !v_cache || !o || !lse || !workspace)
    return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Sq < 1 || Sk < 1) return FATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FATTN_ERR_UNSUPPORTED;
  if (Sq > decode::kMaxSq) return FATTN_ERR_UNSUPPORTED;
  if (dtype != FATTN_FP16 && dtype != FATTN_BF16) return FATTN_ERR_UNSUPPORTED;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) |
                        reinterpret_cast<uintptr_t>(k_cache) |
                        reinterpret_cast<uintptr_t>(v_cache) |
                        reinterpret_cast<uintptr_t>(o) |
                        reinterpret_cast<uintptr_t>(workspace);
  if ((a16 & 15u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0)
    return FATTN_ERR_MISALIGNED;

  DeviceState* ds = nullptr;
  int dev = 0;
  int rc = current_device(&ds, &dev);
  if (rc != kOk) return rc;
  KvPlan plan;
  rc = kvcache_checks(B, H, Sq, Sk, D, ds->sms, &plan);
  if (rc != kOk) return rc;
  if (workspace_bytes < plan.ws_bytes) return FATTN_ERR_INVALID_ARG;

  const size_t bh = (size_t)B * H;
  const size_t qbytes = bh * Sq * D * 2;
  const size_t cbytes = bh * Sk * D * 2;
  const size_t lbytes = bh * Sq * sizeof(float);
  const size_t nbytes = cache_lens ? (size_t)B * sizeof(int) : 0;
  const size_t wbytes = (size_t)plan.ws_bytes;
  const void* ins[4] = {q, k_cache, v_cache, cache_lens};
  const size_t insz[4] = {qbytes, cbytes, cbytes, nbytes};
  const void* outs[3] = {o, lse, workspace};
  const size_t outsz[3] = {qbytes, lbytes, wbytes};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 4; ++j)
      if (insz[j] && overlaps(outs[i], outsz[i], ins[j], insz[j]))
        return FATTN_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (overlaps(outs[i], outsz[i], outs[j], outsz[j])) return FATTN_ERR_INVALID_ARG;
  }
  for (int j = 0; j < 4; ++j)
    if (insz[j] && (rc = check_device_buffer(ins[j], insz[j], dev)) != kOk) return rc;
  for (int i = 0; i < 3; ++i)
    if ((rc = check_device_buffer(outs[i], outsz[i], dev)) != kOk) return rc;

  const bool bf16 = dtype == FATTN_BF16;
  CUtensorMap tm_k, tm_v;
  if (encode_cache(&tm_k, k_cache, Sk, (int)bh, D, bf16) != kOk ||
      encode_cache(&tm_v, v_cache, Sk, (int)bh, D, bf16) != kOk)
    return FATTN_ERR_CUDA;

  decode::DecodeLaunch a;
  a.tm_k = &tm_k;
  a.tm_v = &tm_v;
  decode::DecodeParams& p = a.params;
  p.q = q;
  p.lens = cache_lens;
  p.part_o = static_cast<float*>(workspace);
  p.part_lse = static_cast<float*>(workspace) + plan.records * (size_t)Sq * D;
  p.o = o;
  p.lse = lse;
  p.status = ds->status;
  p.B = B;
  p.H = H;
  p.Sq = Sq;
  p.Sk = Sk;
  p.causal = causal != 0;
  p.n_warps = plan.split_warps;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.timeout_ns = wait_timeout_ns();
  a.grid = plan.grid;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  if (decode::launch(D, bf16, a) != cudaSuccess) {
    cudaGetLastError();
    return FATTN_ERR_LAUNCH;
  }
  return FATTN_OK;
}

FATTN_API int fattn_fwd_fp8(const void* q, const void* k, const void* v, void* o,
                            float* lse, int B, int H, int S, int D, int causal,
                            float scale, float q_scale, float k_scale, float v_scale,
                            int out_dtype, fattn_stream_t stream) {
  // ---- host-side checks, nothing enqueued yet
  if (!q || !k || !v || !o || !lse) return FATTN_ERR_INVALID_ARG;
  for (float x : {scale, q_scale, k_scale, v_scale})
    if (!(x > 0.0f) || !std::isfinite(x)) return FATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S < 1) return FATTN_ERR_INVALID_ARG;
  if (D != 128) return FATTN_ERR_UNSUPPORTED;
  if (out_dtype != FATTN_FP16 && out_dtype != FATTN_BF16) return FATTN_ERR_UNSUPPORTED;
  const long long rows = (long long)B * H * S;
  if (rows > INT_MAX) return FATTN_ERR_TOO_LARGE;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if ((a16 & 15u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return FATTN_ERR_MISALIGNED;
  const size_t ibytes = (size_t)rows * D;      // E4M3
  const size_t obytes = (size_t)rows * D * 2;  // 16-bit output
  const size_t lbytes = (size_t)rows * sizeof(float);
  if (overlaps(o, obytes, q, ibytes) || overlaps(o, obytes, k, ibytes) ||
      overlaps(o, obytes, v, ibytes) || overlaps(lse, lbytes, q, ibytes) ||
      overlaps(lse, lbytes, k, ibytes) || overlaps(lse, lbytes, v, ibytes) ||
      overlaps(lse, lbytes, o, obytes))
    return FATTN_ERR_INVALID_ARG;

  DeviceState* ds = nullptr;
  int dev = 0;
  int rc = current_device(&ds, &dev);
  if (rc != kOk) return rc;
  if ((rc = check_device_buffer(q, ibytes, dev)) != kOk) return rc;
  if ((rc = check_device_buffer(k, ibytes, dev)) != kOk) return rc;
  if ((rc = check_device_buffer(v, ibytes, dev)) != kOk) return rc;
  if ((rc = check_device_buffer(o, obytes, dev)) != kOk) return rc;
  if ((rc = check_device_buffer(lse, lbytes, dev)) != kOk) return rc;

  const int BH = B * H;
  CUtensorMap tm_q, tm_k, tm_v;
  if (encode_bhsd_e4m3(&tm_q, q, S, BH, D) != kOk ||
      encode_bhsd_e4m3(&tm_k, k, S, BH, D) != kOk ||
      encode_bhsd_e4m3(&tm_v, v, S, BH, D) != kOk)
    return FATTN_ERR_CUDA;
  const int units_per_head = (S + 2 * kBM - 1) / (2 * kBM);
  const long long total = (long long)BH * units_per_head;
  if (total > INT_MAX) return FATTN_ERR_TOO_LARGE;

  LaunchArgs a;
  a.tm_q = &tm_q;
  a.tm_k = &tm_k;
  a.tm_v = &tm_v;
  a.params.o = o;
  a.params.lse = lse;
  a.params.status = ds->status;
  a.params.S = S;
  a.params.BH = BH;
  a.params.n_kv_tiles = (S + kBN - 1) / kBN;
  a.params.n_units = units_per_head;
  a.params.total_units = (int)total;
  // scores of the real values: scale * (q_scale Q8) . (k_scale K8)
  a.params.scale_log2 =
      (float)((double)scale * q_scale * k_scale * 1.4426950408889634);
  a.params.o_scale = v_scale;
  a.params.timeout_ns = wait_timeout_ns();
  a.grid = (int)total < ds->sms ? (int)total : ds->sms;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  // as for 16-bit inputs at D = 128: units at run time only when the K and
  // V of all heads exceed one group
  int group = BH;
  bool run_time_units = false;
  if (causal) causal_order(BH, S, D, 1, units_per_head, ds->sms, &group, &run_time_units);
  a.params.sched = run_time_units ? sched_pair(ds, a.stream) : nullptr;
  a.params.group_heads = group;
  if (launch_fwd_fp8_d128(causal != 0, out_dtype == FATTN_BF16, a) != cudaSuccess) {
    cudaGetLastError();
    return FATTN_ERR_LAUNCH;
  }
  return FATTN_OK;
}

FATTN_API int fattn_check_wait_timeout(int timeout_us, fattn_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return FATTN_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  const int rc = current_device(&ds, nullptr);
  if (rc != kOk) return rc;
  wait_check_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      ds->status, (unsigned long long)timeout_us * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return FATTN_ERR_LAUNCH;
  return FATTN_OK;
}

FATTN_API int fattn_last_error(fattn_stream_t stream, int* detail) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FATTN_ERR_CUDA;
  }
  DeviceState* ds = nullptr;
  const int rc = current_device(&ds, nullptr);
  if (rc != kOk) return rc;
  int h[kStatusWords] = {0, 0, 0, 0};
  if (cudaMemcpy(h, ds->status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(ds->status, 0, sizeof(h)) != cudaSuccess) {
    cudaGetLastError();
    return FATTN_ERR_CUDA;
  }
  if (detail) {
    detail[0] = h[1];
    detail[1] = h[2];
  }
  return h[0];
}

FATTN_API int fattn_fwd_kvcache_noalloc(const void* q, const void* k_cache,
                                        const void* v_cache, const int* cache_lens,
                                        void* o, float* lse, int B, int H, int Sq,
                                        int Sk, int D, int causal, float scale,
                                        int dtype, int* status_words,
                                        fattn_stream_t stream) {
  // ---- host-side checks, nothing enqueued yet
  if (!q || !k_cache || !v_cache || !o || !lse) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Sq < 1 || Sk < 1) return FATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FATTN_ERR_UNSUPPORTED;
  if (Sq > decode::kMaxSq) return FATTN_ERR_UNSUPPORTED;
  if (dtype != FATTN_FP16 && dtype != FATTN_BF16) return FATTN_ERR_UNSUPPORTED;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) |
                        reinterpret_cast<uintptr_t>(k_cache) |
                        reinterpret_cast<uintptr_t>(v_cache) |
                        reinterpret_cast<uintptr_t>(o);
  if ((a16 & 15u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(status_words) & 3u) != 0)
    return FATTN_ERR_MISALIGNED;

  NoAllocState* ds = nullptr;
  int dev = 0;
  int rc = noalloc_device(&ds, &dev);
  if (rc != kOk) return rc;
  KvPlan plan;
  rc = kvcache_checks(B, H, Sq, Sk, D, ds->sms, &plan);
  if (rc != kOk) return rc;
  if (plan.ws_bytes > FATTN_NOALLOC_SCRATCH_BYTES) return FATTN_ERR_TOO_LARGE;

  const size_t bh = (size_t)B * H;
  const size_t qbytes = bh * Sq * D * 2;
  const size_t cbytes = bh * Sk * D * 2;
  const size_t lbytes = bh * Sq * sizeof(float);
  const size_t nbytes = cache_lens ? (size_t)B * sizeof(int) : 0;
  const size_t sbytes = status_words ? sizeof(int) * kStatusWords : 0;
  const void* ins[4] = {q, k_cache, v_cache, cache_lens};
  const size_t insz[4] = {qbytes, cbytes, cbytes, nbytes};
  const void* outs[3] = {o, lse, status_words};
  const size_t outsz[3] = {qbytes, lbytes, sbytes};
  for (int i = 0; i < 3; ++i) {
    if (!outsz[i]) continue;
    for (int j = 0; j < 4; ++j)
      if (insz[j] && overlaps(outs[i], outsz[i], ins[j], insz[j]))
        return FATTN_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (outsz[j] && overlaps(outs[i], outsz[i], outs[j], outsz[j]))
        return FATTN_ERR_INVALID_ARG;
  }
  for (int j = 0; j < 4; ++j)
    if (insz[j] && (rc = check_device_buffer(ins[j], insz[j], dev)) != kOk) return rc;
  for (int i = 0; i < 3; ++i)
    if (outsz[i] && (rc = check_device_buffer(outs[i], outsz[i], dev)) != kOk) return rc;

  const bool bf16 = dtype == FATTN_BF16;
  CUtensorMap tm_k, tm_v;
  if (encode_cache(&tm_k, k_cache, Sk, (int)bh, D, bf16) != kOk ||
      encode_cache(&tm_v, v_cache, Sk, (int)bh, D, bf16) != kOk)
    return FATTN_ERR_CUDA;

  decode::DecodeLaunch a;
  a.tm_k = &tm_k;
  a.tm_v = &tm_v;
  decode::DecodeParams& p = a.params;
  p.q = q;
  p.lens = cache_lens;
  p.part_o = static_cast<float*>(ds->scratch);
  p.part_lse = static_cast<float*>(ds->scratch) + plan.records * (size_t)Sq * D;
  p.o = o;
  p.lse = lse;
  p.status = status_words ? status_words : ds->status;
  p.B = B;
  p.H = H;
  p.Sq = Sq;
  p.Sk = Sk;
  p.causal = causal != 0;
  p.n_warps = plan.split_warps;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.timeout_ns = wait_timeout_ns();
  a.grid = plan.grid;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  if (decode::launch(D, bf16, a) != cudaSuccess) {
    cudaGetLastError();
    return FATTN_ERR_LAUNCH;
  }
  return FATTN_OK;
}

}  // extern "C"
