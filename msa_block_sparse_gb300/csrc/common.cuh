// Shared host/device plumbing of libmsa: error reporting, tensor-map encoding,
// per-call tile plans and launch helpers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cstddef>
#include <string>
#include <utility>

#include "../../include/msa.h"

namespace msa {

constexpr int kD = 128;         // head dim
constexpr int kBlock = 128;     // key block (tokens)
constexpr int kTopK = 16;       // selected blocks per query
constexpr int kRopeDim = 64;    // rotated channels

// ------------------------------------------------------------------ host errors

void set_error(const char* fmt, ...);
msa_status_t fail(msa_status_t code, const char* fmt, ...);
msa_status_t check_launch(const char* what);

// Process-unique id (cuCtxGetId) of the calling thread's current CUDA
// context, 0 when none is current.
msa_status_t current_context_id(unsigned long long* id);

// Device address of a file-scope __device__ variable (given by its host-side
// stand-in `symbol`) in the calling thread's current CUDA context, looked up
// with cudaGetSymbolAddress once per (variable, context) and cached.  The key
// is the context's process-unique id (cuCtxGetId), so a context created after
// cudaDeviceReset gets its own lookup instead of a stale address.
msa_status_t symbol_address(const void* symbol, const char* what, void** out);

// Address of the device status word in the current context; MSA_ERR_CUDA
// (nothing enqueued) when it cannot be had.
msa_status_t status_word(uint32_t** out);

// Brackets one kernel launch with CUDA events on `stream` while tracing is on
// (msa_trace_begin / msa_trace_end); does nothing otherwise.
class TraceScope {
 public:
  TraceScope(const char* kernel, cudaStream_t stream);
  ~TraceScope();
  TraceScope(const TraceScope&) = delete;
  TraceScope& operator=(const TraceScope&) = delete;

 private:
  int slot_ = -1;
  cudaStream_t stream_;
};

// ------------------------------------------------------------------ tensor maps

// bf16 tensor with up to 3 dims (dims[0] innermost, contiguous), 128B swizzle.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint32_t* box);
// fp32 tensor, same conventions (128B swizzle: the box's inner extent is 32 floats).
bool make_tmap_f32(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                   const uint32_t* box);
// bf16 tensor of rank 2..5 with explicit byte strides of dims 1.. (multiples of
// 16, in any order), 128B swizzle; dims[0] is contiguous.
bool make_tmap_bf16_strided(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides, const uint32_t* box);

// ------------------------------------------------------------------ workspace

// Bump allocator over the caller's workspace (256-byte aligned pieces).
struct WsCursor {
  uint8_t* base;
  size_t used = 0;
  explicit WsCursor(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    size_t off = (used + 255) & ~size_t(255);
    used = off + count * sizeof(T);
    return base ? reinterpret_cast<T*>(base + off) : nullptr;
  }
};

// ------------------------------------------------------------------ tile plan
// The tiles (sequence s, tile q) of a pack, `tile` consecutive tokens each
// (128 by default: one key block), ordered by q descending (heaviest causal work
// first), then s ascending.  Built on the device from cu_seqlens by `launch_plan`.
struct Plan {
  int2* tiles;      // [max_tiles] (s, q)
  int* num_tiles;   // [1]
  int max_tiles;    // host-side upper bound: T / tile + S
  int tile;         // tokens per tile
};

inline int plan_max_tiles(int T, int S, int tile = kBlock) { return T / tile + S; }
Plan carve_plan(WsCursor& ws, int T, int S, int tile = kBlock);
msa_status_t launch_plan(const Plan& plan, const int32_t* cu_seqlens, int S, int max_seqlen,
                         cudaStream_t stream);

// Launches `kernel` with programmatic stream serialization, so that its launch
// overlaps the tail of the previous kernel on `stream`; the kernel itself
// orders its memory accesses after that kernel with pdl_wait().
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace msa
