// C ABI of libmsa: argument validation, workspace layout, error reporting and
// the per-call tile plan.  The compute kernels live in the other .cu files.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.cuh"

namespace msa {

// ------------------------------------------------------------------ errors

static thread_local char g_last_error[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
}

msa_status_t fail(msa_status_t code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

msa_status_t check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return MSA_OK;
}

// ------------------------------------------------------------------ status word

// [0] status bits, [1] first expired wait (0x80000000 | site id), [2] its block
// (x + y << 20), [3] its thread
__device__ uint32_t g_device_status[4];

namespace {

template <class F>
F driver_fn(const char* name, unsigned int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(p);
}

}  // namespace

// Process-unique id of the calling thread's current context (0 if none).
msa_status_t current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_current = driver_fn<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent", 4000);
    get_id = driver_fn<PFN_cuCtxGetId_v12000>("cuCtxGetId", 12000);
  });
  if (!get_current || !get_id) return fail(MSA_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId unavailable");
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return fail(MSA_ERR_CUDA, "cuCtxGetCurrent failed");
  *id = 0;
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return fail(MSA_ERR_CUDA, "cuCtxGetId failed");
  return MSA_OK;
}

namespace {

std::mutex g_symbol_mu;
std::map<std::pair<const void*, unsigned long long>, void*> g_symbol_cache;

}  // namespace

msa_status_t symbol_address(const void* symbol, const char* what, void** out) {
  unsigned long long ctx = 0;
  msa_status_t st = current_context_id(&ctx);
  if (st != MSA_OK) return st;
  std::lock_guard<std::mutex> lk(g_symbol_mu);
  if (ctx != 0) {
    auto it = g_symbol_cache.find(std::make_pair(symbol, ctx));
    if (it != g_symbol_cache.end()) {
      *out = it->second;
      return MSA_OK;
    }
  }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, symbol);   // makes the primary context current if none is
  if (e != cudaSuccess || p == nullptr)
    return fail(MSA_ERR_CUDA, "cudaGetSymbolAddress(%s): %s", what, cudaGetErrorString(e));
  if (ctx == 0) {
    st = current_context_id(&ctx);
    if (st != MSA_OK) return st;
  }
  if (ctx != 0) g_symbol_cache[std::make_pair(symbol, ctx)] = p;
  *out = p;
  return MSA_OK;
}

msa_status_t status_word(uint32_t** out) {
  void* p = nullptr;
  msa_status_t st = symbol_address(&g_device_status, "status word", &p);
  *out = static_cast<uint32_t*>(p);
  return st;
}

// ------------------------------------------------------------------ device

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

size_t device_l2_bytes() {
  static size_t cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev);
    cached[dev] = n > 0 ? static_cast<size_t>(n) : 1;
  }
  return cached[dev];
}

msa_status_t ensure_smem_ptr(const void* kernel, size_t bytes, const char* name) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(MSA_ERR_CUDA, "cudaGetDevice failed");
  std::lock_guard<std::mutex> lk(mu);
  size_t& have = done[std::make_pair(kernel, dev)];
  if (have < bytes) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(bytes)) != cudaSuccess)
      return fail(MSA_ERR_CUDA, "%s: %zu bytes of dynamic shared memory refused", name, bytes);
    have = bytes;
  }
  return MSA_OK;
}

// ------------------------------------------------------------------ tracing

namespace {
struct TraceRec {
  const char* name;
  cudaEvent_t start, stop;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace_pool;   // events are created once and reused
size_t g_trace_used = 0;
}  // namespace

TraceScope::TraceScope(const char* kernel, cudaStream_t stream) : stream_(stream) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (!g_trace_on) return;
  if (g_trace_used == g_trace_pool.size()) {
    TraceRec r{nullptr, nullptr, nullptr};
    if (cudaEventCreate(&r.start) != cudaSuccess || cudaEventCreate(&r.stop) != cudaSuccess)
      return;
    g_trace_pool.push_back(r);
  }
  slot_ = static_cast<int>(g_trace_used++);
  g_trace_pool[slot_].name = kernel;
  cudaEventRecord(g_trace_pool[slot_].start, stream_);
}

TraceScope::~TraceScope() {
  if (slot_ < 0) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  cudaEventRecord(g_trace_pool[slot_].stop, stream_);
}

// ------------------------------------------------------------------ tensor maps

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

static bool make_tmap(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                      uint64_t elem_bytes, int rank, const uint64_t* dims, const uint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[3], gstride[2];
  cuuint32_t bdim[3], estr[3] = {1, 1, 1};
  uint64_t stride = elem_bytes;
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    if (i > 0) gstride[i - 1] = stride;
    stride *= dims[i];
  }
  CUresult r = fn(map, dtype, rank, const_cast<void*>(base), gdim, gstride, bdim, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint32_t* box) {
  return make_tmap(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rank, dims, box);
}

bool make_tmap_f32(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                   const uint32_t* box) {
  return make_tmap(map, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, rank, dims, box);
}

bool make_tmap_bf16_strided(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides, const uint32_t* box) {
  auto fn = encode_fn();
  if (!fn || rank < 2 || rank > 5) return false;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estr[5] = {1, 1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    if (i > 0) gstride[i - 1] = strides[i - 1];
  }
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gdim,
                  gstride, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ tile plan

// One CTA.  nb(s) = ceil(len_s / tile) tiles per sequence; tiles are listed with
// qb descending, s ascending.  cnt[q] = #{s : nb(s) > q}; start[q] = sum of
// cnt[q'] for q' > q; thread q then appends (s, q) for every qualifying s in
// order, so the list is deterministic.  Both suffix sums are block-wide scans
// over the entries taken from the top (1024 per pass, a running carry between
// passes); nb(s) is kept in shared memory when it fits beside them.
__host__ __device__ constexpr bool plan_keeps_nb(int S, int max_nb) {
  return (2 * (max_nb + 1) + S) * 4 <= 48 * 1024;
}

// inclusive scan of v over the CTA; *total = the sum over the CTA
__device__ __forceinline__ int block_incl_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += x;
  }
  if (lane == 31) warp_sums[wp] = v;
  __syncthreads();
  if (wp == 0) {
    int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += x;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  v += wp > 0 ? warp_sums[wp - 1] : 0;
  *total = warp_sums[nw - 1];
  __syncthreads();                          // warp_sums may be reused
  return v;
}

__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ cu, int S,
                                                    int tile, int max_nb,
                                                    int2* __restrict__ tiles,
                                                    int* __restrict__ num_tiles, int max_tiles,
                                                    uint32_t* status) {
  pdl_enter();
  extern __shared__ int sh[];
  int* cnt = sh;                     // [max_nb + 1]
  int* start = sh + max_nb + 1;      // [max_nb + 1]
  int* nbs = sh + 2 * (max_nb + 1);  // [S] when it fits
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x;
  const bool keep = plan_keeps_nb(S, max_nb);
  for (int q = tid; q <= max_nb; q += blockDim.x) cnt[q] = 0;
  __syncthreads();
  auto nb_of = [&](int s) {
    const int len = cu[s + 1] - cu[s];
    const int nb = (len + tile - 1) / tile;
    return len < 0 ? 0 : (nb > max_nb ? max_nb : nb);
  };
  for (int s = tid; s < S; s += blockDim.x) {
    const int len = cu[s + 1] - cu[s];
    if (len < 0 || (len + tile - 1) / tile > max_nb) atomicOr(status, kStatusBounds);
    const int nb = nb_of(s);
    if (keep) nbs[s] = nb;
    if (nb > 0) atomicAdd(&cnt[nb - 1], 1);   // histogram of nb - 1
  }
  __syncthreads();
  // entry i of a pass is q = max_nb - 1 - i: the running inclusive scan is the
  // suffix sum cnt[q] = #{s : nb(s) - 1 >= q}; a second running scan of those,
  // less the entry itself, is start[q] = sum_{q' > q} cnt[q']
  int carry_c = 0, carry_s = 0;
  for (int base = 0; base < max_nb; base += blockDim.x) {
    const int q = max_nb - 1 - (base + tid);
    int tot_c, tot_s;
    const int c = carry_c + block_incl_scan(q >= 0 ? cnt[q] : 0, warp_sums, &tot_c);
    const int st = carry_s + block_incl_scan(q >= 0 ? c : 0, warp_sums, &tot_s);
    if (q >= 0) {
      cnt[q] = c;
      start[q] = st - c;
    }
    carry_c += tot_c;
    carry_s += tot_s;
  }
  if (tid == 0) {
    *num_tiles = carry_s < max_tiles ? carry_s : max_tiles;
    if (carry_s > max_tiles) atomicOr(status, kStatusBounds);
  }
  __syncthreads();
  for (int qq = tid; qq < max_nb; qq += blockDim.x) {
    int pos = start[qq];
    for (int s = 0; s < S; ++s) {
      const int nb = keep ? nbs[s] : nb_of(s);
      if (nb > qq && pos < max_tiles) tiles[pos++] = make_int2(s, qq);
    }
  }
}

Plan carve_plan(WsCursor& ws, int T, int S, int tile) {
  Plan p;
  p.tile = tile;
  p.max_tiles = plan_max_tiles(T, S, tile);
  p.tiles = ws.take<int2>(p.max_tiles);
  p.num_tiles = ws.take<int>(1);
  return p;
}

msa_status_t launch_plan(const Plan& plan, const int32_t* cu_seqlens, int S, int max_seqlen,
                         cudaStream_t stream) {
  int max_nb = (max_seqlen + plan.tile - 1) / plan.tile;
  size_t smem = (2 * (max_nb + 1) + (plan_keeps_nb(S, max_nb) ? S : 0)) * sizeof(int);
  uint32_t* sw = nullptr;
  if (msa_status_t e = status_word(&sw); e != MSA_OK) return e;
  {
    TraceScope trace_("plan_kernel", stream);
    launch_pdl(plan_kernel, 1, 1024, smem, stream, cu_seqlens, S, plan.tile, max_nb, plan.tiles,
        plan.num_tiles, plan.max_tiles, sw);
  }
  return check_launch("plan_kernel");
}

}  // namespace msa

using namespace msa;

// ====================================================================== C ABI

static msa_status_t check_pack(const int32_t* cu, int S, int T, int max_seqlen) {
  if (!cu || !aligned16(cu)) return fail(MSA_ERR_INVALID_ARG, "cu_seqlens null or misaligned");
  if (S < 1) return fail(MSA_ERR_INVALID_ARG, "S must be >= 1 (got %d)", S);
  if (T < 1) return fail(MSA_ERR_INVALID_ARG, "T must be >= 1 (got %d)", T);
  if (max_seqlen < 1 || max_seqlen > T)
    return fail(MSA_ERR_INVALID_ARG, "max_seqlen %d outside [1, T=%d]", max_seqlen, T);
  if (max_seqlen > kMaxSeqlen)
    return fail(MSA_ERR_UNSUPPORTED, "max_seqlen %d above the supported %d", max_seqlen,
                kMaxSeqlen);
  return MSA_OK;
}

#define MSA_REQUIRE_PTR(p)                                                            \
  do {                                                                                \
    if (!(p) || !aligned16(p))                                                        \
      return fail(MSA_ERR_INVALID_ARG, "%s is null or not 16-byte aligned", #p);      \
  } while (0)

#define MSA_TRY(expr)                 \
  do {                                \
    msa_status_t _s = (expr);         \
    if (_s != MSA_OK) return _s;      \
  } while (0)

extern "C" {

int msa_abi_version(void) { return MSA_ABI_VERSION; }

msa_status_t msa_trace_begin(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_used = 0;
  g_trace_on = true;
  return MSA_OK;
}

msa_status_t msa_trace_end(char* json, size_t cap) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = false;
  std::map<std::string, std::pair<long, double>> agg;
  std::vector<std::string> order;
  for (size_t i = 0; i < g_trace_used; ++i) {
    const TraceRec& r = g_trace_pool[i];
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      return fail(MSA_ERR_CUDA, "trace: event timing failed");
    auto it = agg.find(r.name);
    if (it == agg.end()) {
      order.push_back(r.name);
      agg[r.name] = {1, ms};
    } else {
      it->second.first += 1;
      it->second.second += ms;
    }
  }
  std::string out = "{";
  for (size_t i = 0; i < order.size(); ++i) {
    char buf[256];
    const auto& v = agg[order[i]];
    snprintf(buf, sizeof(buf), "%s\"%s\": {\"launches\": %ld, \"ms\": %.6f}", i ? ", " : "",
             order[i].c_str(), v.first, v.second);
    out += buf;
  }
  out += "}";
  g_trace_used = 0;
  if (json && cap > 0) {
    const size_t n = out.size() < cap - 1 ? out.size() : cap - 1;
    memcpy(json, out.data(), n);
    json[n] = '\0';
  }
  return MSA_OK;
}

const char* msa_last_error(void) { return g_last_error; }

msa_status_t msa_check_status(msa_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MSA_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
  uint32_t* sw = nullptr;
  if (msa_status_t st = status_word(&sw); st != MSA_OK) return st;
  uint32_t v[4] = {0, 0, 0, 0};
  e = cudaMemcpy(v, sw, sizeof(v), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(sw, 0, sizeof(v));
  if (e != cudaSuccess) return fail(MSA_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (v[0] & kStatusTimeout)
    return fail(MSA_ERR_TIMEOUT,
                "a kernel wait ran out (status %u; first: wait site %u, block (%u, %u), thread %u)",
                v[0], v[1] & 0x7fffffffu, v[2] & 0xfffffu, v[2] >> 20, v[3]);
  if (v[0] & kStatusBounds) return fail(MSA_ERR_BOUNDS, "an index was out of range (status %u)", v[0]);
  return MSA_OK;
}

// One thread waits on an mbarrier that nothing arrives on: the bounded wait
// runs out, records site 65535 in the status word and returns.
__global__ void selftest_wait_kernel(uint32_t* status) {
  pdl_enter();
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, status, 0xFFFFu);
}

msa_status_t msa_selftest_wait(msa_stream_t stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* sw = nullptr;
  if (msa_status_t e = status_word(&sw); e != MSA_OK) return e;
  {
    TraceScope trace_("selftest_wait_kernel", st);
    launch_pdl(selftest_wait_kernel, 1, 32, 0, st, sw);
  }
  return check_launch("selftest_wait_kernel");
}

// ---------------------------------------------------------------- prologue

static msa_status_t check_rope(int rope_dim, float rope_base, float eps) {
  if (rope_dim != kRopeDim)
    return fail(MSA_ERR_UNSUPPORTED, "rope_dim must be %d (got %d)", kRopeDim, rope_dim);
  if (!(rope_base > 1.0f)) return fail(MSA_ERR_INVALID_ARG, "rope_base must be > 1");
  if (!(eps >= 0.0f)) return fail(MSA_ERR_INVALID_ARG, "eps must be >= 0");
  return MSA_OK;
}

msa_status_t msa_qk_norm_rope(const void* x, void* y, int T, int H, const void* w,
                              const int32_t* cu_seqlens, int S, int rope_dim, float rope_base,
                              float eps, msa_stream_t stream) {
  MSA_REQUIRE_PTR(x);
  MSA_REQUIRE_PTR(y);
  MSA_REQUIRE_PTR(w);
  MSA_TRY(check_pack(cu_seqlens, S, T, T));
  MSA_TRY(check_rope(rope_dim, rope_base, eps));
  if (H < 1) return fail(MSA_ERR_INVALID_ARG, "H must be >= 1");
  PrologueJob job{static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y),
                  static_cast<const __nv_bfloat16*>(w), H};
  return launch_prologue(&job, 1, cu_seqlens, S, T, rope_base, eps,
                         static_cast<cudaStream_t>(stream));
}

msa_status_t msa_qk_norm_rope4(const void* q, void* q_out, int Hq, const void* k, void* k_out,
                               int Hkv, const void* q_idx, void* q_idx_out, const void* k_idx,
                               void* k_idx_out, int Hi, const void* w_q, const void* w_k,
                               const void* w_qi, const void* w_ki, const int32_t* cu_seqlens,
                               int S, int T, int rope_dim, float rope_base, float eps,
                               msa_stream_t stream) {
  MSA_REQUIRE_PTR(q);
  MSA_REQUIRE_PTR(k);
  MSA_REQUIRE_PTR(q_idx);
  MSA_REQUIRE_PTR(k_idx);
  MSA_REQUIRE_PTR(q_out);
  MSA_REQUIRE_PTR(k_out);
  MSA_REQUIRE_PTR(q_idx_out);
  MSA_REQUIRE_PTR(k_idx_out);
  MSA_REQUIRE_PTR(w_q);
  MSA_REQUIRE_PTR(w_k);
  MSA_REQUIRE_PTR(w_qi);
  MSA_REQUIRE_PTR(w_ki);
  MSA_TRY(check_pack(cu_seqlens, S, T, T));
  MSA_TRY(check_rope(rope_dim, rope_base, eps));
  if (Hq < 1 || Hkv < 1 || Hi < 1) return fail(MSA_ERR_INVALID_ARG, "head counts must be >= 1");
  using bf = __nv_bfloat16;
  PrologueJob jobs[4] = {
      {static_cast<const bf*>(q), static_cast<bf*>(q_out), static_cast<const bf*>(w_q), Hq},
      {static_cast<const bf*>(k), static_cast<bf*>(k_out), static_cast<const bf*>(w_k), Hkv},
      {static_cast<const bf*>(q_idx), static_cast<bf*>(q_idx_out), static_cast<const bf*>(w_qi),
       Hi},
      {static_cast<const bf*>(k_idx), static_cast<bf*>(k_idx_out), static_cast<const bf*>(w_ki),
       Hi}};
  return launch_prologue(jobs, 4, cu_seqlens, S, T, rope_base, eps,
                         static_cast<cudaStream_t>(stream));
}

size_t msa_qk_norm_rope_bwd_workspace_size(int T, int H) {
  if (T < 1 || H < 1) return 0;
  return prologue_bwd_workspace_floats(T) * sizeof(float);
}

msa_status_t msa_qk_norm_rope_bwd(const void* x, const void* dy, void* dx, float* dw, int T,
                                  int H, const void* w, const int32_t* cu_seqlens, int S,
                                  int rope_dim, float rope_base, float eps, void* workspace,
                                  size_t workspace_bytes, msa_stream_t stream) {
  MSA_REQUIRE_PTR(x);
  MSA_REQUIRE_PTR(dy);
  MSA_REQUIRE_PTR(dx);
  MSA_REQUIRE_PTR(dw);
  MSA_REQUIRE_PTR(w);
  MSA_REQUIRE_PTR(workspace);
  MSA_TRY(check_pack(cu_seqlens, S, T, T));
  MSA_TRY(check_rope(rope_dim, rope_base, eps));
  if (H < 1) return fail(MSA_ERR_INVALID_ARG, "H must be >= 1");
  if (workspace_bytes < msa_qk_norm_rope_bwd_workspace_size(T, H))
    return fail(MSA_ERR_INVALID_ARG, "workspace too small");
  using bf = __nv_bfloat16;
  return launch_prologue_bwd(static_cast<const bf*>(x), static_cast<const bf*>(dy),
                             static_cast<bf*>(dx), dw, static_cast<const bf*>(w), H, cu_seqlens,
                             S, T, rope_base, eps, static_cast<float*>(workspace),
                             static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- index select

size_t msa_index_select_workspace_size(int T, int S, int Hi, int max_seqlen) {
  (void)max_seqlen;
  if (T < 1 || S < 1 || Hi < 1) return 0;
  WsCursor ws(nullptr);
  carve_select_workspace(ws, T, S, Hi);
  return ws.used + 256;
}

msa_status_t msa_index_select(const void* q_idx, const void* k_idx, const int32_t* cu_seqlens,
                              int S, int T, int Hi, int max_seqlen, int topk, int32_t* sel,
                              void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  return msa_index_select_ex(q_idx, k_idx, cu_seqlens, S, T, Hi, max_seqlen, topk, 0, sel,
                             workspace, workspace_bytes, stream);
}

msa_status_t msa_index_select_ex(const void* q_idx, const void* k_idx, const int32_t* cu_seqlens,
                                 int S, int T, int Hi, int max_seqlen, int topk, int n_init,
                                 int32_t* sel, void* workspace, size_t workspace_bytes,
                                 msa_stream_t stream) {
  MSA_REQUIRE_PTR(q_idx);
  MSA_REQUIRE_PTR(k_idx);
  MSA_REQUIRE_PTR(sel);
  MSA_REQUIRE_PTR(workspace);
  MSA_TRY(check_pack(cu_seqlens, S, T, max_seqlen));
  if (topk != kTopK) return fail(MSA_ERR_UNSUPPORTED, "topk must be %d (got %d)", kTopK, topk);
  if (Hi < 1) return fail(MSA_ERR_INVALID_ARG, "Hi must be >= 1");
  if (n_init < 0 || n_init > kTopK - 1)
    return fail(MSA_ERR_INVALID_ARG, "n_init %d outside [0, %d]", n_init, kTopK - 1);
  if (workspace_bytes < msa_index_select_workspace_size(T, S, Hi, max_seqlen))
    return fail(MSA_ERR_INVALID_ARG, "workspace too small");
  WsCursor ws(workspace);
  SelWorkspace w = carve_select_workspace(ws, T, S, Hi);
  return launch_index_select(q_idx, k_idx, cu_seqlens, S, T, Hi, max_seqlen, n_init, w, sel,
                             static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- sparse forward

static msa_status_t check_heads(int Hq, int Hkv) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
    return fail(MSA_ERR_INVALID_ARG, "Hq (%d) must be a positive multiple of Hkv (%d)", Hq, Hkv);
  int G = Hq / Hkv;
  if (G > 128 || (128 % G) != 0)
    return fail(MSA_ERR_UNSUPPORTED, "Hq/Hkv = %d must divide 128", G);
  return MSA_OK;
}

size_t msa_sparse_attn_fwd_workspace_size(int T, int S, int Hq, int Hkv, int max_seqlen) {
  (void)Hq;
  (void)max_seqlen;
  if (T < 1 || S < 1 || Hkv < 1) return 0;
  WsCursor ws(nullptr);
  carve_fwd_workspace(ws, T, S, Hkv);
  return ws.used + 256;
}

static msa_status_t sparse_attn_fwd(const void* q, const void* k, const void* v,
                                    const int32_t* sel, const int32_t* cu_seqlens, int S, int T,
                                    int Hq, int Hkv, int max_seqlen, float scale, void* o,
                                    float* lse, void* workspace, size_t workspace_bytes,
                                    const FwdClear& clear, msa_stream_t stream) {
  MSA_REQUIRE_PTR(q);
  MSA_REQUIRE_PTR(k);
  MSA_REQUIRE_PTR(v);
  MSA_REQUIRE_PTR(sel);
  MSA_REQUIRE_PTR(o);
  MSA_REQUIRE_PTR(lse);
  MSA_REQUIRE_PTR(workspace);
  MSA_TRY(check_pack(cu_seqlens, S, T, max_seqlen));
  MSA_TRY(check_heads(Hq, Hkv));
  if (!(scale > 0.0f)) return fail(MSA_ERR_INVALID_ARG, "scale must be > 0");
  if (workspace_bytes < msa_sparse_attn_fwd_workspace_size(T, S, Hq, Hkv, max_seqlen))
    return fail(MSA_ERR_INVALID_ARG, "workspace too small");
  WsCursor ws(workspace);
  FwdWorkspace fw = carve_fwd_workspace(ws, T, S, Hkv);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MSA_TRY(launch_plan(fw.plan, cu_seqlens, S, max_seqlen, st));
  return launch_sparse_fwd(q, k, v, sel, cu_seqlens, S, T, Hq, Hkv, max_seqlen, scale, fw, o,
                           lse, clear, st);
}

msa_status_t msa_sparse_attn_fwd(const void* q, const void* k, const void* v, const int32_t* sel,
                                 const int32_t* cu_seqlens, int S, int T, int Hq, int Hkv,
                                 int max_seqlen, float scale, void* o, float* lse,
                                 void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  return sparse_attn_fwd(q, k, v, sel, cu_seqlens, S, T, Hq, Hkv, max_seqlen, scale, o, lse,
                         workspace, workspace_bytes, FwdClear{}, stream);
}

msa_status_t msa_sparse_attn_fwd_train(const void* q, const void* k, const void* v,
                                       const int32_t* sel, const int32_t* cu_seqlens, int S,
                                       int T, int Hq, int Hkv, int max_seqlen, float scale,
                                       void* o, float* lse, void* workspace,
                                       size_t workspace_bytes, void* bwd_workspace,
                                       size_t bwd_workspace_bytes, msa_stream_t stream) {
  MSA_REQUIRE_PTR(bwd_workspace);
  MSA_TRY(check_heads(Hq, Hkv));
  if (T < 1 || S < 1 || max_seqlen < 1)
    return fail(MSA_ERR_INVALID_ARG, "bad sizes T=%d S=%d max_seqlen=%d", T, S, max_seqlen);
  if (bwd_workspace_bytes < msa_sparse_attn_bwd_workspace_size(T, S, Hq, Hkv, max_seqlen))
    return fail(MSA_ERR_INVALID_ARG, "backward workspace too small");
  WsCursor bws(bwd_workspace);
  const BwdWorkspace bw = carve_bwd_workspace(bws, T, S, Hq, Hkv, max_seqlen);
  // the three fp32 accumulators are carved back to back (multiples of 16
  // bytes); the item counters after them are cleared as ints
  FwdClear clear;
  clear.ptr = bw.dq_acc;
  clear.bytes = reinterpret_cast<uint8_t*>(bw.dv_acc + static_cast<size_t>(T) * Hkv * kD) -
                reinterpret_cast<uint8_t*>(bw.dq_acc);
  clear.ints = bw.item_ctr;
  clear.nints = Hkv;
  return sparse_attn_fwd(q, k, v, sel, cu_seqlens, S, T, Hq, Hkv, max_seqlen, scale, o, lse,
                         workspace, workspace_bytes, clear, stream);
}

// ---------------------------------------------------------------- sparse backward

size_t msa_sparse_attn_bwd_workspace_size(int T, int S, int Hq, int Hkv, int max_seqlen) {
  if (T < 1 || S < 1 || Hq < 1 || Hkv < 1 || max_seqlen < 1) return 0;
  WsCursor ws(nullptr);
  carve_bwd_workspace(ws, T, S, Hq, Hkv, max_seqlen);
  return ws.used + 256;
}

static msa_status_t sparse_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                                    const void* dout, const float* lse, const int32_t* sel,
                                    const int32_t* cu_seqlens, int S, int T, int Hq, int Hkv,
                                    int max_seqlen, float scale, void* dq, void* dk, void* dv,
                                    void* workspace, size_t workspace_bytes, bool clear_acc,
                                    msa_stream_t stream) {
  MSA_REQUIRE_PTR(q);
  MSA_REQUIRE_PTR(k);
  MSA_REQUIRE_PTR(v);
  MSA_REQUIRE_PTR(o);
  MSA_REQUIRE_PTR(dout);
  MSA_REQUIRE_PTR(lse);
  MSA_REQUIRE_PTR(sel);
  MSA_REQUIRE_PTR(dq);
  MSA_REQUIRE_PTR(dk);
  MSA_REQUIRE_PTR(dv);
  MSA_REQUIRE_PTR(workspace);
  MSA_TRY(check_pack(cu_seqlens, S, T, max_seqlen));
  MSA_TRY(check_heads(Hq, Hkv));
  if (!(scale > 0.0f)) return fail(MSA_ERR_INVALID_ARG, "scale must be > 0");
  if (workspace_bytes < msa_sparse_attn_bwd_workspace_size(T, S, Hq, Hkv, max_seqlen))
    return fail(MSA_ERR_INVALID_ARG, "workspace too small");
  WsCursor ws(workspace);
  BwdWorkspace bw = carve_bwd_workspace(ws, T, S, Hq, Hkv, max_seqlen);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return launch_sparse_bwd(q, k, v, o, dout, lse, sel, cu_seqlens, S, T, Hq, Hkv, max_seqlen,
                           scale, bw, dq, dk, dv, clear_acc, st);
}

msa_status_t msa_sparse_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                                 const void* dout, const float* lse, const int32_t* sel,
                                 const int32_t* cu_seqlens, int S, int T, int Hq, int Hkv,
                                 int max_seqlen, float scale, void* dq, void* dk, void* dv,
                                 void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  return sparse_attn_bwd(q, k, v, o, dout, lse, sel, cu_seqlens, S, T, Hq, Hkv, max_seqlen,
                         scale, dq, dk, dv, workspace, workspace_bytes, true, stream);
}

msa_status_t msa_sparse_attn_bwd_prepare(int T, int S, int Hq, int Hkv, int max_seqlen,
                                         void* workspace, size_t workspace_bytes,
                                         msa_stream_t stream) {
  MSA_REQUIRE_PTR(workspace);
  if (T < 1 || S < 1 || max_seqlen < 1 || max_seqlen > T)
    return fail(MSA_ERR_INVALID_ARG, "bad sizes T=%d S=%d max_seqlen=%d", T, S, max_seqlen);
  MSA_TRY(check_heads(Hq, Hkv));
  if (workspace_bytes < msa_sparse_attn_bwd_workspace_size(T, S, Hq, Hkv, max_seqlen))
    return fail(MSA_ERR_INVALID_ARG, "workspace too small");
  WsCursor ws(workspace);
  BwdWorkspace bw = carve_bwd_workspace(ws, T, S, Hq, Hkv, max_seqlen);
  return launch_bwd_clear(bw, Hkv, static_cast<cudaStream_t>(stream));
}

msa_status_t msa_sparse_attn_bwd_prepared(const void* q, const void* k, const void* v,
                                          const void* o, const void* dout, const float* lse,
                                          const int32_t* sel, const int32_t* cu_seqlens, int S,
                                          int T, int Hq, int Hkv, int max_seqlen, float scale,
                                          void* dq, void* dk, void* dv, void* workspace,
                                          size_t workspace_bytes, msa_stream_t stream) {
  return sparse_attn_bwd(q, k, v, o, dout, lse, sel, cu_seqlens, S, T, Hq, Hkv, max_seqlen,
                         scale, dq, dk, dv, workspace, workspace_bytes, false, stream);
}

// ---------------------------------------------------------------- narrow blocks

static msa_status_t check_qsa(const int32_t* cu, int S, int T, int Hq, int Hkv, int topk,
                              int max_seqlen, float scale) {
  MSA_TRY(check_pack(cu, S, T, max_seqlen));
  if (Hkv < 1 || Hq != 12 * Hkv)
    return fail(MSA_ERR_UNSUPPORTED, "narrow-block attention needs Hq = 12 Hkv (got %d, %d)",
                Hq, Hkv);
  if (topk < 1 || topk > kQsaMaxTopk)
    return fail(MSA_ERR_INVALID_ARG, "topk %d outside [1, %d]", topk, kQsaMaxTopk);
  if (max_seqlen > kQsaMaxSeqlen)
    return fail(MSA_ERR_UNSUPPORTED, "max_seqlen %d above the supported %d for 4-token blocks",
                max_seqlen, kQsaMaxSeqlen);
  if (!(scale > 0.0f)) return fail(MSA_ERR_INVALID_ARG, "scale must be > 0");
  return MSA_OK;
}

size_t msa_qsa_attn_fwd_workspace_size(int T, int S, int Hq, int Hkv, int max_seqlen) {
  (void)Hq;
  if (T < 1 || S < 1 || Hkv < 1 || max_seqlen < 1 || max_seqlen > kQsaMaxSeqlen) return 0;
  WsCursor ws(nullptr);
  carve_qsa_fwd_workspace(ws, T, S, Hkv, max_seqlen);
  return ws.used + 256;
}

msa_status_t msa_qsa_attn_fwd(const void* q, const void* k, const void* v, const int32_t* sel,
                              const int32_t* cu_seqlens, int S, int T, int Hq, int Hkv, int topk,
                              int max_seqlen, float scale, void* o, float* lse, void* workspace,
                              size_t workspace_bytes, msa_stream_t stream) {
  MSA_REQUIRE_PTR(q);
  MSA_REQUIRE_PTR(k);
  MSA_REQUIRE_PTR(v);
  MSA_REQUIRE_PTR(sel);
  MSA_REQUIRE_PTR(o);
  MSA_REQUIRE_PTR(lse);
  MSA_REQUIRE_PTR(workspace);
  MSA_TRY(check_qsa(cu_seqlens, S, T, Hq, Hkv, topk, max_seqlen, scale));
  if (workspace_bytes < msa_qsa_attn_fwd_workspace_size(T, S, Hq, Hkv, max_seqlen))
    return fail(MSA_ERR_INVALID_ARG, "workspace too small");
  WsCursor ws(workspace);
  QsaFwdWorkspace fw = carve_qsa_fwd_workspace(ws, T, S, Hkv, max_seqlen);
  return launch_qsa_fwd(q, k, v, sel, cu_seqlens, S, T, Hq, Hkv, topk, max_seqlen, scale, fw, o,
                        lse, static_cast<cudaStream_t>(stream));
}

size_t msa_qsa_attn_bwd_workspace_size(int T, int S, int Hq, int Hkv, int max_seqlen) {
  if (T < 1 || S < 1 || Hq < 1 || Hkv < 1 || max_seqlen < 1 || max_seqlen > kQsaMaxSeqlen)
    return 0;
  WsCursor ws(nullptr);
  carve_qsa_bwd_workspace(ws, T, S, Hq, Hkv, max_seqlen);
  return ws.used + 256;
}

msa_status_t msa_qsa_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, const int32_t* sel,
                              const int32_t* cu_seqlens, int S, int T, int Hq, int Hkv, int topk,
                              int max_seqlen, float scale, void* dq, void* dk, void* dv,
                              void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  MSA_REQUIRE_PTR(q);
  MSA_REQUIRE_PTR(k);
  MSA_REQUIRE_PTR(v);
  MSA_REQUIRE_PTR(o);
  MSA_REQUIRE_PTR(dout);
  MSA_REQUIRE_PTR(lse);
  MSA_REQUIRE_PTR(sel);
  MSA_REQUIRE_PTR(dq);
  MSA_REQUIRE_PTR(dk);
  MSA_REQUIRE_PTR(dv);
  MSA_REQUIRE_PTR(workspace);
  MSA_TRY(check_qsa(cu_seqlens, S, T, Hq, Hkv, topk, max_seqlen, scale));
  if (workspace_bytes < msa_qsa_attn_bwd_workspace_size(T, S, Hq, Hkv, max_seqlen))
    return fail(MSA_ERR_INVALID_ARG, "workspace too small");
  WsCursor ws(workspace);
  QsaBwdWorkspace bw = carve_qsa_bwd_workspace(ws, T, S, Hq, Hkv, max_seqlen);
  return launch_qsa_bwd(q, k, v, o, dout, lse, sel, cu_seqlens, S, T, Hq, Hkv, topk, max_seqlen,
                        scale, bw, dq, dk, dv, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- decode

size_t msa_decode_step_workspace_size(int B, int Hq, int Hkv, int max_pages) {
  if (B < 1 || Hq < 1 || Hkv < 1 || max_pages < 1) return 0;
  WsCursor ws(nullptr);
  carve_decode_workspace(ws, B, Hq, Hkv, max_pages);
  return ws.used + 256;
}

msa_status_t msa_decode_step(const void* q, const void* q_idx, const void* k_cache,
                             const void* v_cache, const void* kidx_cache,
                             const int32_t* block_table, const int32_t* cache_lens, int B, int Hq,
                             int Hkv, int num_pages, int max_pages, float scale, void* o,
                             int32_t* sel_out, void* workspace, size_t workspace_bytes,
                             msa_stream_t stream) {
  return msa_decode_step_ex(q, q_idx, k_cache, v_cache, kidx_cache, block_table, cache_lens, B,
                            Hq, Hkv, num_pages, max_pages, scale, 0, o, sel_out, workspace,
                            workspace_bytes, stream);
}

msa_status_t msa_decode_step_ex(const void* q, const void* q_idx, const void* k_cache,
                                const void* v_cache, const void* kidx_cache,
                                const int32_t* block_table, const int32_t* cache_lens, int B,
                                int Hq, int Hkv, int num_pages, int max_pages, float scale,
                                int n_init, void* o, int32_t* sel_out, void* workspace,
                                size_t workspace_bytes, msa_stream_t stream) {
  MSA_REQUIRE_PTR(q);
  MSA_REQUIRE_PTR(q_idx);
  MSA_REQUIRE_PTR(k_cache);
  MSA_REQUIRE_PTR(v_cache);
  MSA_REQUIRE_PTR(kidx_cache);
  MSA_REQUIRE_PTR(block_table);
  MSA_REQUIRE_PTR(cache_lens);
  MSA_REQUIRE_PTR(o);
  MSA_REQUIRE_PTR(workspace);
  if (sel_out && !aligned16(sel_out))
    return fail(MSA_ERR_INVALID_ARG, "sel_out is not 16-byte aligned");
  if (B < 1 || num_pages < 1 || max_pages < 1)
    return fail(MSA_ERR_INVALID_ARG, "B, num_pages and max_pages must be >= 1");
  if (max_pages > kMaxSeqlen / kBlock)
    return fail(MSA_ERR_UNSUPPORTED, "max_pages %d above the supported %d", max_pages,
                kMaxSeqlen / kBlock);
  MSA_TRY(check_heads(Hq, Hkv));
  if (Hq / Hkv != 16) return fail(MSA_ERR_UNSUPPORTED, "decode needs Hq/Hkv = 16");
  if (!(scale > 0.0f)) return fail(MSA_ERR_INVALID_ARG, "scale must be > 0");
  if (n_init < 0 || n_init > kTopK - 1)
    return fail(MSA_ERR_INVALID_ARG, "n_init %d outside [0, %d]", n_init, kTopK - 1);
  if (workspace_bytes < msa_decode_step_workspace_size(B, Hq, Hkv, max_pages))
    return fail(MSA_ERR_INVALID_ARG, "workspace too small");
  WsCursor ws(workspace);
  DecodeWorkspace dw = carve_decode_workspace(ws, B, Hq, Hkv, max_pages);
  return launch_decode(q, q_idx, k_cache, v_cache, kidx_cache, block_table, cache_lens, B, Hq, Hkv,
                       num_pages, max_pages, scale, n_init, o, sel_out, dw,
                       static_cast<cudaStream_t>(stream));
}

msa_status_t msa_decode_append(const void* q, const void* q_idx, const void* k, const void* v,
                               const void* k_idx, const void* w_q, const void* w_qi,
                               const void* w_k, const void* w_ki, void* k_cache, void* v_cache,
                               void* kidx_cache, const int32_t* block_table,
                               const int32_t* cache_lens, int B, int Hq, int Hkv, int num_pages,
                               int max_pages, int rope_dim, float rope_base, float eps,
                               void* q_out, void* q_idx_out, msa_stream_t stream) {
  MSA_REQUIRE_PTR(q);
  MSA_REQUIRE_PTR(q_idx);
  MSA_REQUIRE_PTR(k);
  MSA_REQUIRE_PTR(v);
  MSA_REQUIRE_PTR(k_idx);
  MSA_REQUIRE_PTR(w_q);
  MSA_REQUIRE_PTR(w_qi);
  MSA_REQUIRE_PTR(w_k);
  MSA_REQUIRE_PTR(w_ki);
  MSA_REQUIRE_PTR(k_cache);
  MSA_REQUIRE_PTR(v_cache);
  MSA_REQUIRE_PTR(kidx_cache);
  MSA_REQUIRE_PTR(block_table);
  MSA_REQUIRE_PTR(cache_lens);
  MSA_REQUIRE_PTR(q_out);
  MSA_REQUIRE_PTR(q_idx_out);
  if (B < 1 || num_pages < 1 || max_pages < 1)
    return fail(MSA_ERR_INVALID_ARG, "B, num_pages and max_pages must be >= 1");
  if (max_pages > kMaxSeqlen / kBlock)
    return fail(MSA_ERR_UNSUPPORTED, "max_pages %d above the supported %d", max_pages,
                kMaxSeqlen / kBlock);
  MSA_TRY(check_heads(Hq, Hkv));
  MSA_TRY(check_rope(rope_dim, rope_base, eps));
  using bf = __nv_bfloat16;
  DecodeAppendJob j;
  j.q = static_cast<const bf*>(q);
  j.q_idx = static_cast<const bf*>(q_idx);
  j.k = static_cast<const bf*>(k);
  j.v = static_cast<const bf*>(v);
  j.k_idx = static_cast<const bf*>(k_idx);
  j.w_q = static_cast<const bf*>(w_q);
  j.w_qi = static_cast<const bf*>(w_qi);
  j.w_k = static_cast<const bf*>(w_k);
  j.w_ki = static_cast<const bf*>(w_ki);
  j.q_out = static_cast<bf*>(q_out);
  j.q_idx_out = static_cast<bf*>(q_idx_out);
  j.k_cache = static_cast<bf*>(k_cache);
  j.v_cache = static_cast<bf*>(v_cache);
  j.kidx_cache = static_cast<bf*>(kidx_cache);
  j.Hq = Hq;
  j.Hkv = Hkv;
  return launch_decode_append(j, block_table, cache_lens, B, num_pages, max_pages, rope_base,
                              eps, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
