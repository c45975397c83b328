// zero_reduce_norm_noalloc: the reduce + overflow + squared-norm pass over W
// flat gradient buffers, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running while a CUDA graph
// is being captured elsewhere in the process, allocator-less embeddings that
// own every byte of device memory up front, or hosts that forbid the library
// from growing its footprint after start-up. This entry point therefore keeps
// its only scratch -- one fp64 partial and one overflow flag per chunk of
// kNaChunk elements, and a completion counter -- in a file-scope
// `static __device__` array. Every GPU that loads the library holds that
// array (about 768 KB) until the process exits.
//
// The caller passes all inputs and outputs. Host code must not hand the
// array's name to a kernel: on the host that name is only a stand-in, not a
// device address. The device address belongs to one CUDA context (each
// context loads its own copy of the module), so it is looked up with
// cudaGetSymbolAddress on the first call made in each context and cached
// under that context's unique ID (cuCtxGetId): a context created after
// cudaDeviceReset, or one the caller made current through the driver API,
// gets its own lookup instead of a stale address.
#include <cuda.h>  // CUcontext / CUresult types; the two driver calls are resolved at run time
#include <mutex>

#include "k_reduce.cuh"
#include "zero.h"

namespace zg {

constexpr int64_t kNaChunk = 65536;      // elements per partial
constexpr int64_t kNaMaxChunks = 65536;  // partials the array holds -> n <= 2^32 elements
constexpr size_t kNaCounterBytes = 256;
constexpr size_t kNaScratchBytes =
    kNaCounterBytes + kNaMaxChunks * sizeof(double) + kNaMaxChunks * sizeof(unsigned);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaScratchBytes];

struct NaArgs {
  const void* grads[kMaxWorld];
  int world;
  int64_t n;
  int64_t n_chunks;
  void* reduced;           // comm dtype, n elements, or nullptr
  double* norm_sq_out;
  int32_t* overflow_out;
  unsigned char* scratch;  // device address of g_noalloc_scratch
};

template <typename GT, typename CT>
__global__ void __launch_bounds__(kThreads) k_reduce_norm_noalloc(const __grid_constant__ NaArgs a) {
  __shared__ double s_red[kThreads / 32];
  __shared__ unsigned s_or[kThreads / 32];
  __shared__ bool s_last;
  unsigned* counter = reinterpret_cast<unsigned*>(a.scratch);
  double* part = reinterpret_cast<double*>(a.scratch + kNaCounterBytes);
  unsigned* flags = reinterpret_cast<unsigned*>(a.scratch + kNaCounterBytes + kNaMaxChunks * 8);
  CT* out = static_cast<CT*>(a.reduced);

  for (int64_t c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
    const int64_t lo = c * kNaChunk;
    const int64_t hi_end = lo + kNaChunk < a.n ? lo + kNaChunk : a.n;
    const int64_t nvec = (hi_end - lo) >> 3;
    float hi = 0.0f, lo_c = 0.0f;
    double big = 0.0;
    unsigned bad = 0u;
    for (int64_t v = threadIdx.x; v < nvec; v += kThreads) {
      const int64_t i = lo + v * 8;
      float s[8];
      load8(static_cast<const GT*>(a.grads[0]) + i, s);
      for (int w = 1; w < a.world; ++w) add8(static_cast<const GT*>(a.grads[w]) + i, s);
      Pack8<CT> rc;
      float rf[8];
      float ss = 0.0f;
      bool fin = true;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        rc.e[j] = DT<CT>::from_f32(s[j]);
        rf[j] = DT<CT>::to_f32(rc.e[j]);
        fin = fin && DT<CT>::finite_bits(rc.e[j]);
        ss = __fmaf_rn(rf[j], rf[j], ss);
      }
      if (!fin) bad = 1u;
      add_group(ss, hi, lo_c, big, rf);
      if (out != nullptr) store8_raw(out + i, rc);
    }
    const int64_t tail0 = lo + nvec * 8;
    if (threadIdx.x < hi_end - tail0) {
      const int64_t i = tail0 + threadIdx.x;
      float sum = load1(static_cast<const GT*>(a.grads[0]), i);
      for (int w = 1; w < a.world; ++w) sum = __fadd_rn(sum, load1(static_cast<const GT*>(a.grads[w]), i));
      const CT rc = DT<CT>::from_f32(sum);
      const double rf = (double)DT<CT>::to_f32(rc);
      if (!DT<CT>::finite_bits(rc)) bad = 1u;
      big += rf * rf;
      if (out != nullptr) out[i] = rc;
    }
    const double total = block_sum<kThreads>((double)hi + (double)lo_c + big, s_red);
    const unsigned any = block_or<kThreads>(bad, s_or);
    if (threadIdx.x == 0) {
      part[c] = total;
      flags[c] = any;
    }
  }

  // The last block to finish sums the partials in chunk order.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  double acc = 0.0;
  unsigned any = 0u;
  for (int64_t c = threadIdx.x; c < a.n_chunks; c += kThreads) {
    acc += __ldcg(part + c);
    any |= __ldcg(flags + c);
  }
  const double total = block_sum<kThreads>(acc, s_red);
  const unsigned ovf = block_or<kThreads>(any, s_or);
  if (threadIdx.x == 0) {
    *a.norm_sq_out = total;
    *a.overflow_out = ovf ? 1 : 0;
    *counter = 0u;  // leave the array ready for the next call
  }
}

template <typename GT>
static const void* na_kernel_g(int comm_dtype) {
  switch (comm_dtype) {
    case kF32: return reinterpret_cast<const void*>(&k_reduce_norm_noalloc<GT, float>);
    case kF16: return reinterpret_cast<const void*>(&k_reduce_norm_noalloc<GT, __half>);
    case kBF16: return reinterpret_cast<const void*>(&k_reduce_norm_noalloc<GT, __nv_bfloat16>);
    default: return nullptr;
  }
}

static const void* na_kernel(int grad_dtype, int comm_dtype) {
  switch (grad_dtype) {
    case kF32: return na_kernel_g<float>(comm_dtype);
    case kF16: return na_kernel_g<__half>(comm_dtype);
    case kBF16: return na_kernel_g<__nv_bfloat16>(comm_dtype);
    default: return nullptr;
  }
}

// Per-context set-up: the array's device address in that context and the
// device's SM count, keyed by the context's process-unique ID. The table is
// small and reused round-robin; IDs are never reused, so an entry of a
// destroyed context can never be matched again.
struct NaContext {
  unsigned long long ctx_id = 0;  // 0: empty slot
  unsigned char* scratch = nullptr;
  int sms = 0;
};
constexpr int kNaMaxContexts = 64;
static NaContext g_na_ctx[kNaMaxContexts];
static int g_na_next = 0;
static std::mutex g_na_mutex;

typedef CUresult (*NaCtxGetCurrent)(CUcontext*);
typedef CUresult (*NaCtxGetId)(CUcontext, unsigned long long*);
static NaCtxGetCurrent g_get_current = nullptr;
static NaCtxGetId g_get_id = nullptr;

// The unique ID of the context current on this thread (caller holds
// g_na_mutex). A thread on which the runtime has not yet made a context
// current gets the device's primary context first, as any runtime call would.
static int na_current_context(unsigned long long* id) {
  if (g_get_current == nullptr || g_get_id == nullptr) {
    cudaDriverEntryPointQueryResult q1, q2;
    void* f1 = nullptr;
    void* f2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) !=
            cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess)
      return zero_internal_fail(ZERO_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId not available");
    g_get_current = reinterpret_cast<NaCtxGetCurrent>(f1);
    g_get_id = reinterpret_cast<NaCtxGetId>(f2);
  }
  CUcontext c = nullptr;
  if (g_get_current(&c) != CUDA_SUCCESS)
    return zero_internal_fail(ZERO_ERR_CUDA, "cuCtxGetCurrent failed");
  if (c == nullptr) {  // no context yet: let the runtime bind the primary one
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return zero_internal_fail(ZERO_ERR_CUDA, cudaGetErrorString(e));
    if (g_get_current(&c) != CUDA_SUCCESS || c == nullptr)
      return zero_internal_fail(ZERO_ERR_CUDA, "no CUDA context is current");
  }
  if (g_get_id(c, id) != CUDA_SUCCESS || *id == 0)
    return zero_internal_fail(ZERO_ERR_CUDA, "cuCtxGetId failed");
  return ZERO_OK;
}

}  // namespace zg

using namespace zg;

extern "C" int zero_reduce_norm_noalloc(const void* const* grads, int world, int64_t n,
                                        int grad_dtype, int comm_dtype, void* reduced_out,
                                        double* norm_sq_out, int32_t* overflow_out, void* stream) {
  if (grads == nullptr || norm_sq_out == nullptr || overflow_out == nullptr)
    return zero_internal_fail(ZERO_ERR_INVALID, "grads, norm_sq_out and overflow_out are required");
  if (world < 1 || world > kMaxWorld)
    return zero_internal_fail(ZERO_ERR_INVALID, "world outside 1..64");
  if (n < 0) return zero_internal_fail(ZERO_ERR_INVALID, "n must not be negative");
  if (n > kNaChunk * kNaMaxChunks)
    return zero_internal_fail(ZERO_ERR_INVALID,
                              "n exceeds the no-alloc scratch capacity (2^32 elements)");
  const int comm = comm_dtype < 0 ? grad_dtype : comm_dtype;
  const void* f = na_kernel(grad_dtype, comm);
  if (f == nullptr) return zero_internal_fail(ZERO_ERR_INVALID, "bad grad_dtype or comm_dtype");
  NaArgs a{};
  for (int w = 0; w < world; ++w) {
    if (grads[w] == nullptr || (reinterpret_cast<uintptr_t>(grads[w]) & 15u) != 0)
      return zero_internal_fail(ZERO_ERR_INVALID, "grads[w] NULL or not 16-byte aligned");
    a.grads[w] = grads[w];
  }
  if ((reinterpret_cast<uintptr_t>(reduced_out) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(norm_sq_out) & 7u) != 0 ||
      (reinterpret_cast<uintptr_t>(overflow_out) & 3u) != 0)
    return zero_internal_fail(ZERO_ERR_INVALID, "misaligned output pointer");

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return zero_internal_fail(ZERO_ERR_CUDA, cudaGetErrorString(e));
  NaContext d;
  {
    std::lock_guard<std::mutex> lock(g_na_mutex);
    unsigned long long id = 0;
    const int rc = na_current_context(&id);
    if (rc != ZERO_OK) return rc;
    int hit = -1;
    for (int i = 0; i < kNaMaxContexts; ++i)
      if (g_na_ctx[i].ctx_id == id) hit = i;
    if (hit < 0) {  // first call in this context: look the array up here
      NaContext c;
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return zero_internal_fail(ZERO_ERR_CUDA, cudaGetErrorString(e));
      e = cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return zero_internal_fail(ZERO_ERR_CUDA, cudaGetErrorString(e));
      c.ctx_id = id;
      c.scratch = static_cast<unsigned char*>(p);
      hit = g_na_next;
      g_na_next = (g_na_next + 1) % kNaMaxContexts;
      g_na_ctx[hit] = c;
    }
    d = g_na_ctx[hit];
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n == 0) {
    e = cudaMemsetAsync(norm_sq_out, 0, sizeof(double), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(overflow_out, 0, sizeof(int32_t), s);
    return e == cudaSuccess ? ZERO_OK : zero_internal_fail(ZERO_ERR_CUDA, cudaGetErrorString(e));
  }
  a.world = world;
  a.n = n;
  a.n_chunks = (n + kNaChunk - 1) / kNaChunk;
  a.reduced = reduced_out;
  a.norm_sq_out = norm_sq_out;
  a.overflow_out = overflow_out;
  a.scratch = d.scratch;
  // The completion counter must start at zero (a call cut short could leave it set).
  e = cudaMemsetAsync(d.scratch, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return zero_internal_fail(ZERO_ERR_CUDA, cudaGetErrorString(e));
  const int64_t want = (int64_t)d.sms * 4;
  const int grid = (int)(a.n_chunks < want ? a.n_chunks : want);
  void* args[] = {&a};
  e = cudaLaunchKernel(f, dim3(grid), dim3(kThreads), args, 0, s);
  if (e != cudaSuccess) return zero_internal_fail(ZERO_ERR_CUDA, cudaGetErrorString(e));
  return ZERO_OK;
}
