// Library runtime: per-device status word, launch context, TMA descriptor encoding,
// status queries, the bounded-wait probe and the host RoPE-table helper.
#include <atomic>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace llama {

// One status word per device (this is a per-device variable: each device that loads
// the module has its own copy).  Kernels record the first error with atomicCAS(0, code).
// Words 2.. hold the record that the first timed-out wait leaves (see mbar_wait_slow).
constexpr int kStatusWords = 2 + 2 * kTimeoutRecordFields;
__device__ __align__(16) int g_status_word[kStatusWords];

namespace {

std::atomic<int*> g_status_addr[kMaxDevices];
std::atomic<int> g_num_sms[kMaxDevices];
std::atomic<uint64_t> g_launches{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace

int make_ctx(void* stream, Ctx* c) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LLAMA_ERR_CUDA;
  int* st = g_status_addr[dev].load(std::memory_order_acquire);
  if (st == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return LLAMA_ERR_CUDA;
    st = static_cast<int*>(p);
    g_status_addr[dev].store(st, std::memory_order_release);
  }
  int sms = g_num_sms[dev].load(std::memory_order_acquire);
  if (sms == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return LLAMA_ERR_CUDA;
    g_num_sms[dev].store(sms, std::memory_order_release);
  }
  c->stream = static_cast<cudaStream_t>(stream);
  c->device = dev;
  c->num_sms = sms;
  c->status = st;
  return LLAMA_OK;
}

namespace {
// Optional per-thread trace: caller-owned CUDA events recorded on the launch stream
// once when tracing starts and after every kernel launch (for timing kernel by kernel).
thread_local void* const* t_events = nullptr;
thread_local int t_n = 0;
thread_local int t_next = 0;
}  // namespace

bool trace_active() { return t_events != nullptr; }

int after_launch(const Ctx& c) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  const bool ok = cudaGetLastError() == cudaSuccess;
  if (t_events != nullptr && t_next < t_n)
    cudaEventRecord(static_cast<cudaEvent_t>(t_events[t_next++]), c.stream);
  return ok ? LLAMA_OK : LLAMA_ERR_CUDA;
}

bool make_tmap_2d(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr || base == nullptr || cols == 0 || rows == 0) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_3d(CUtensorMap* tm, const void* base, uint64_t n0, uint64_t n1, uint64_t n2, uint64_t s1,
                  uint64_t s2, uint32_t box1) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr || base == nullptr || n0 == 0 || n1 == 0 || n2 == 0) return false;
  const cuuint64_t dims[3] = {n0, n1, n2};
  const cuuint64_t strides[2] = {s1 * 2, s2 * 2};
  const cuuint32_t box[3] = {64, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// One thread waits on an mbarrier that nothing arrives at; the bounded wait gives up.
__global__ void wait_probe_kernel(uint64_t budget_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_test(smem_u32(&bar), 0))
      mbar_wait_slow(smem_u32(&bar), 0, status, &abort_flag, budget_ns);
  }
  __syncthreads();
}

}  // namespace
}  // namespace llama

using namespace llama;

extern "C" {

int llama_get_device_status(void* cuda_stream) {
  Ctx c;
  int rc = make_ctx(cuda_stream, &c);
  if (rc != LLAMA_OK) return rc;
  if (cudaStreamSynchronize(c.stream) != cudaSuccess) return LLAMA_ERR_CUDA;
  int v = 0;
  const int zero = 0;
  if (cudaMemcpy(&v, c.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (cudaMemcpy(c.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return LLAMA_ERR_CUDA;
  return v;
}

const char* llama_status_string(int s) {
  switch (s) {
    case LLAMA_OK: return "ok";
    case LLAMA_ERR_INVALID_ARG: return "invalid argument";
    case LLAMA_ERR_UNSUPPORTED: return "unsupported shape";
    case LLAMA_ERR_CUDA: return "CUDA error";
    case LLAMA_ERR_TIMEOUT: return "device-side wait timed out";
    case LLAMA_ERR_DEVICE_BOUNDS: return "device-side index out of range";
    case LLAMA_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of llama_attention_decode_static";
    default: return "unknown status";
  }
}

int llama_debug_timeout_record(int64_t* out, int32_t n) {
  if (out == nullptr || n <= 0) return LLAMA_ERR_INVALID_ARG;
  Ctx c;
  int rc = make_ctx(nullptr, &c);
  if (rc != LLAMA_OK) return rc;
  long long rec[kTimeoutRecordFields];
  if (cudaMemcpy(rec, c.status + 2, sizeof(rec), cudaMemcpyDeviceToHost) != cudaSuccess) return LLAMA_ERR_CUDA;
  for (int i = 0; i < n && i < kTimeoutRecordFields; ++i) out[i] = rec[i];
  return LLAMA_OK;
}

int llama_debug_wait_probe(uint64_t budget_ns, void* cuda_stream) {
  Ctx c;
  int rc = make_ctx(cuda_stream, &c);
  if (rc != LLAMA_OK) return rc;
  const uint64_t cap = 10ull * 1000ull * 1000ull * 1000ull;
  wait_probe_kernel<<<1, 32, 0, c.stream>>>(budget_ns < cap ? budget_ns : cap, c.status);
  return after_launch(c);
}

uint64_t llama_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int llama_trace_begin(void* const* events, int32_t n_events, void* cuda_stream) {
  if (events == nullptr || n_events < 1) return LLAMA_ERR_INVALID_ARG;
  t_events = events;
  t_n = n_events;
  t_next = 0;
  if (cudaEventRecord(static_cast<cudaEvent_t>(events[t_next++]), static_cast<cudaStream_t>(cuda_stream)) !=
      cudaSuccess)
    return LLAMA_ERR_CUDA;
  return LLAMA_OK;
}

int32_t llama_trace_end(void) {
  const int n = t_next;
  t_events = nullptr;
  t_n = t_next = 0;
  return n;
}

int llama_rope_tables(double base, int32_t head_dim, int32_t max_pos, float* cos_host, float* sin_host) {
  if (cos_host == nullptr || sin_host == nullptr || head_dim <= 0 || (head_dim & 1) || max_pos <= 0 ||
      !(base > 0.0))
    return LLAMA_ERR_INVALID_ARG;
  const int half = head_dim / 2;
  for (int i = 0; i < half; ++i) {
    const double theta = std::pow(base, -2.0 * static_cast<double>(i) / static_cast<double>(head_dim));
    for (int p = 0; p < max_pos; ++p) {
      const double a = static_cast<double>(p) * theta;
      cos_host[static_cast<size_t>(p) * half + i] = static_cast<float>(std::cos(a));
      sin_host[static_cast<size_t>(p) * half + i] = static_cast<float>(std::sin(a));
    }
  }
  return LLAMA_OK;
}

}  // extern "C"
