// Block-sparse attention backward ("#4581", "Kernel tuning": dQ and dK/dV of
// the block-sparse kernel; "MiniMax-M3.1-Flash", 5.4 "Notable quirks": the
// indexer is frozen, so the selection is a constant here).
//
// KV-major schedule.  A work item is (KV head g, key block b of sequence s, a
// 256-position window of candidate query positions).  Items are listed window
// by window, so the items running at any moment add into dQ rows of a few
// windows only and the fp32 dQ accumulator lines stay in L2.  Persistent CTAs
// (one per SM and KV head share) claim the items from a counter, so that a CTA
// that drew short items takes more; the last fifth of the list (the last third
// when the dQ accumulator is within twice L2) is claimed largest first (the
// order the last CTA of bwd_lists_kernel writes) so that the CTAs finish
// together.  Per item the CTA holds
// K_b and V_b in shared memory and streams the window's query tokens that
// selected b, in ascending order, in half-chunks of 4 tokens x G = 16 heads =
// 64 columns.  A pre-pass (bwd_lists_kernel) lists, per item, those tokens
// (one thread per candidate, ballot compaction); another (bwd_delta_kernel,
// whose CTA 0 also lists the items) packs (lse log2 e,
// Delta) per query row.
//   producers (warp 0: K_b / V_b and the even half-chunks; warp 10: the odd
//            ones; one warp alone cannot issue the copies fast enough): per
//            token one 4 KB tensor load of Q, one of dO (a 5-D tensor map that
//            lays the 16 heads out as the operands need them) and one 128-byte
//            bulk copy of (lse, Delta), into a 4-stage ring
//   MMA (warp 1): S^T = K_b Q^T, dP^T = V_b dO^T -> TMEM slot u & 1;
//            dV += P^T dO (P^T read from TMEM), dK += dS^T Q (after which the
//            stage is free), dQ^T = K_b^T dS^T (both operands MN-major) into
//            the dP^T columns
//   compute (warps 2..9: warpgroup z takes the half-chunks u with u & 1 == z;
//            thread = key row): P^T = exp2(S^T scale log2e - lse log2e),
//            causally masked, packed to bf16 into TMEM; dS^T = P^T (dP^T -
//            Delta) to shared memory, with P^T read back from TMEM (the bf16
//            values dV uses) and -Delta fetched from shared memory while dP^T
//            is computed; then the dQ^T rows are added into the
//            fp32 dQ accumulator with reductions straight from registers (a
//            warp covers 32 consecutive floats of a row); at the end of an item
//            warpgroup 0 adds dK, warpgroup 1 dV into their accumulators.
// A last kernel scales and converts the accumulators to bf16.
#include "kernels.cuh"

namespace msa {

namespace {

constexpr int kGroupThreads = 128;          // a compute warpgroup
// warp 0 TMA (even half-chunks, K/V), warp 1 MMA, warps 2..9 compute (two
// warpgroups), warp 10 TMA (odd half-chunks): one TMA-issuing warp cannot keep
// up with one 4 KB copy per token and tensor
constexpr int kBwdThreads = 64 + 2 * kGroupThreads + 32;
constexpr int kLoaderWarp1 = 2 + 2 * kGroupThreads / 32;
constexpr int kTile = 128 * 128 * 2;
constexpr int kHalf = kTile / 2;
constexpr int kHc = 64;                     // columns of a half-chunk: 4 tokens x 16 heads
constexpr int kHcTok = 4;
constexpr int kStages = 4;
// Claimed item ids pass from the claiming producer to the other roles through a
// ring of slots; each slot is read by the second loader, the MMA issuer and the
// 8 compute warps before it is reused.
constexpr int kItemSlots = 4;
constexpr int kItemReaders = 1 + 1 + 8;
constexpr int kTokBytes = 16 * kD * 2;      // Q (or dO) rows of one token: 4 KB
constexpr int kStageBytes = 2 * kHcTok * kTokBytes;   // Q then dO of a half-chunk: 32 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kIdescS = idesc_bf16(128, kHc, false, false);    // S^T, dP^T (N = 64)
constexpr uint32_t kIdescKM = idesc_bf16(128, 128, false, true);    // dV, dK: B MN-major
constexpr uint32_t kIdescQ = idesc_bf16(128, kHc, true, true);      // dQ^T: both MN-major
// TMEM columns: dV, dK accumulators, then two slots of (S^T | P^T, dP^T | dQ^T)
constexpr uint32_t kColDV = 0, kColDK = 128, kColSlot = 256;

// A token's Q (or dO) image: 32 rows of 128 B, row = 16 (head / 8) + 8 (D half)
// + head % 8, 128B-swizzled.  Column n = 16 token + head of a half-chunk then
// lies in 8-row group n / 8 at 2048 (n / 8) bytes, its D halves 1024 bytes
// apart: a K-major operand with group stride 2048, or an MN-major one with
// D-chunk stride 1024 and K-group stride 2048.
struct BwdSmem {
  uint8_t k[kTile];
  uint8_t v[kTile];
  uint8_t dst[2][kHc * 128 * 2];        // dS^T of each slot: 128 keys x 64 columns
  uint8_t stage[kStages][kStageBytes];  // Q then dO token images
  float lsd[kStages][2 * kHc];          // per token: -lse log2 e of its 16 heads, then -Delta
  int tok[kStages][kHcTok];
  uint64_t kv_full, kv_empty;
  uint64_t ld_full[kStages], ld_empty[kStages];
  uint64_t s_full[2], dp_full[2], p_full[2], ds_full[2], dv_done[2], dq_full[2], dq_free[2];
  uint64_t acc_full, acc_free;
  uint64_t item_full[kItemSlots], item_empty[kItemSlots];
  int item_id[kItemSlots];              // claimed item of the slot; -1: none left
  uint32_t tmem_base;
};
static_assert(sizeof(BwdSmem) <= 232448, "backward shared memory above the 227 KB limit");

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

}  // namespace

// ---------------------------------------------------------------- items

// Run by one whole CTA (CTA 0 of the Delta kernel, whose other work it
// overlaps).  Pairs (window w, sequence s) in w-major order; pair (w, s) holds
// the key blocks b that some query of window w can select: 128 b < min(len,
// (w+1) W).  Each becomes an item (s, b, first position, end position) of that
// window.  A sequence longer than max_seqlen (or of negative length) is
// flagged in the status word and clipped.  Also clears the per-KV-head
// arrival counters of bwd_lists_kernel.
__device__ __forceinline__ void build_items(const int32_t* __restrict__ cu, int S,
                                            int max_seqlen, int num_windows,
                                            int4* __restrict__ items,
                                            int* __restrict__ num_items, int max_items,
                                            int* __restrict__ lists_done, int Hkv,
                                            uint32_t* status) {
  __shared__ int warp_sums[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  for (int g = threadIdx.x; g < Hkv; g += blockDim.x) lists_done[g] = 0;
  __syncthreads();
  const long long npairs = static_cast<long long>(num_windows) * S;
  for (long long base = 0; base < npairs; base += blockDim.x) {
    const long long pi = base + threadIdx.x;
    int s = 0, w = 0, len = 0, cnt = 0;
    if (pi < npairs) {
      w = static_cast<int>(pi / S);
      s = static_cast<int>(pi % S);
      len = cu[s + 1] - cu[s];
      if (len < 0 || len > max_seqlen) {
        if (w == 0) atomicOr(status, kStatusBounds);
        len = len < 0 ? 0 : max_seqlen;
      }
      const int w0 = w * kBwdSegment;
      if (len > w0) {
        const int hi = min(len, w0 + kBwdSegment);
        cnt = (hi + kBlock - 1) / kBlock;
      }
    }
    int incl = cnt;
    const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += x;
    }
    if (lane == 31) warp_sums[wp] = incl;
    __syncthreads();
    if (wp == 0) {
      int ws = (lane < static_cast<int>(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, ws, d);
        if (lane >= d) ws += x;
      }
      warp_sums[lane] = ws;
    }
    __syncthreads();
    const int off = carry + (wp > 0 ? warp_sums[wp - 1] : 0) + incl - cnt;
    const int w0 = w * kBwdSegment;
    for (int b = 0; b < cnt; ++b) {
      const int idx = off + b;
      if (idx < max_items)
        items[idx] = make_int4(s, b, max(b * kBlock, w0), min(len, w0 + kBwdSegment));
      else
        atomicOr(status, kStatusBounds);
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = off + cnt;
    __syncthreads();
  }
  if (threadIdx.x == 0) *num_items = min(carry, max_items);
}

// ---------------------------------------------------------------- token lists

// Claim order of one KV head's items, written by the last CTA of that head to
// finish its lists.  The first n - n / tail_div items keep their window-major
// order (concurrent items add into the dQ rows of a few windows, which keeps
// the dQ accumulator lines in L2); the rest follow by half-chunk count,
// largest first, so that the last items claimed are short and the CTAs finish
// together.  Order within equal counts is unspecified.
constexpr int kMaxHalfChunks = kBwdSegment / 4;

// gridDim.x CTAs of kBwdSegment threads per KV head (blockIdx.y), grid-striding
// over the items: thread t checks candidate position first + t; the matches
// are compacted in ascending order into the item's list.  The CTA that
// finishes last for its KV head (arrival counter, cleared by build_items)
// then writes that head's claim order.
__global__ void __launch_bounds__(kBwdSegment) bwd_lists_kernel(
    const int32_t* __restrict__ cu, const int32_t* __restrict__ sel,
    const int4* __restrict__ items, const int* __restrict__ num_items, int Hkv,
    int* __restrict__ lists, int* __restrict__ list_len, int* __restrict__ lists_done,
    int max_items, int* __restrict__ order, int tail_div) {
  pdl_enter();
  static_assert(kBwdSegment == 256, "one thread per candidate position");
  __shared__ int warp_cnt[kBwdSegment / 32];
  __shared__ int hist[kMaxHalfChunks + 1], start[kMaxHalfChunks + 1];
  __shared__ int last;
  const int n = *num_items;
  const int g = blockIdx.y;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int it = blockIdx.x; it < n; it += gridDim.x) {
    const int4 item = items[it];
    const int s = item.x, b = item.y;
    const int p = item.z + static_cast<int>(threadIdx.x);
    bool hit = false;
    if (p < item.w) {
      const int4* row = reinterpret_cast<const int4*>(
          sel + (static_cast<size_t>(cu[s] + p) * Hkv + g) * kTopK);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int4 v = __ldg(row + c);
        hit |= (v.x == b) | (v.y == b) | (v.z == b) | (v.w == b);
      }
    }
    const uint32_t m = __ballot_sync(0xffffffffu, hit);
    if (lane == 0) warp_cnt[w] = __popc(m);
    __syncthreads();
    int off = 0, total = 0;
#pragma unroll
    for (int i = 0; i < kBwdSegment / 32; ++i) {
      off += (i < w) ? warp_cnt[i] : 0;
      total += warp_cnt[i];
    }
    const size_t li = static_cast<size_t>(it) * Hkv + g;
    if (hit) lists[li * kBwdSegment + off + __popc(m & ((1u << lane) - 1u))] = p;
    if (threadIdx.x == 0) list_len[li] = total;
    __syncthreads();
  }
  // the last CTA of this KV head: every list_len of the head is written
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(lists_done + g, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int k = n - n / tail_div;
  int* ord = order + static_cast<size_t>(g) * max_items;
  for (int i = threadIdx.x; i <= kMaxHalfChunks; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    if (i < k) {
      ord[i] = i;
    } else {
      const int nh = min((__ldcg(list_len + static_cast<size_t>(i) * Hkv + g) + 3) / 4,
                         kMaxHalfChunks);
      atomicAdd(&hist[nh], 1);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = k;
    for (int c = kMaxHalfChunks; c >= 0; --c) {
      start[c] = acc;
      acc += hist[c];
    }
  }
  __syncthreads();
  for (int i = k + static_cast<int>(threadIdx.x); i < n; i += blockDim.x) {
    const int nh = min((__ldcg(list_len + static_cast<size_t>(i) * Hkv + g) + 3) / 4,
                       kMaxHalfChunks);
    ord[atomicAdd(&start[nh], 1)] = i;
  }
}

// ---------------------------------------------------------------- Delta

// For query row (t, 16 g + j): lsd[32 (t Hkv + g) + j] = -lse log2 e and
// lsd[32 (t Hkv + g) + 16 + j] = -sum_d dout o (= -Delta).  16 lanes per row
// (16-byte loads), kDeltaRows rows per thread with all loads issued first.
constexpr int kDeltaRows = 2;
__global__ void __launch_bounds__(256) bwd_delta_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
    const float* __restrict__ lse, float* __restrict__ lsd, size_t rows,
    const int32_t* __restrict__ cu, int S, int max_seqlen, int num_windows,
    int4* __restrict__ items, int* __restrict__ num_items, int max_items,
    int* __restrict__ lists_done, int Hkv, uint32_t* status) {
  pdl_enter();
  if (blockIdx.x == 0)
    build_items(cu, S, max_seqlen, num_windows, items, num_items, max_items, lists_done, Hkv,
                status);
  const int sub = threadIdx.x & 15;
  const size_t row0 =
      (static_cast<size_t>(blockIdx.x) * (blockDim.x >> 4) + (threadIdx.x >> 4)) * kDeltaRows;
  uint4 a[kDeltaRows], b[kDeltaRows];
  float ls[kDeltaRows];
#pragma unroll
  for (int i = 0; i < kDeltaRows; ++i) {
    const size_t row = row0 + i;
    ls[i] = 0.f;
    if (row < rows) {
      a[i] = __ldcs(reinterpret_cast<const uint4*>(o + row * kD) + sub);
      b[i] = __ldcs(reinterpret_cast<const uint4*>(dout + row * kD) + sub);
      if (sub == 0) ls[i] = __ldg(lse + row);
    }
  }
#pragma unroll
  for (int i = 0; i < kDeltaRows; ++i) {
    const size_t row = row0 + i;
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[i]);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b[i]);
    float acc = 0.f;
    if (row < rows) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 x = __bfloat1622float2(a2[j]);
        const float2 y = __bfloat1622float2(b2[j]);
        acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
      }
    }
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (sub == 0 && row < rows) {
      const size_t j = row & 15, base = (row - j) * 2 + j;
      lsd[base] = -ls[i] * kLog2e;
      lsd[base + 16] = -acc;
    }
  }
}

// ---------------------------------------------------------------- convert

// dq = scale dq_acc, dk = scale dk_acc, dv = dv_acc to bf16 in one launch:
// thread i converts 8 elements; the first nq8 groups are dQ, then dK, then dV.
__global__ void bwd_convert_kernel(const float* __restrict__ dq_acc,
                                   const float* __restrict__ dk_acc,
                                   const float* __restrict__ dv_acc,
                                   __nv_bfloat16* __restrict__ dq, __nv_bfloat16* __restrict__ dk,
                                   __nv_bfloat16* __restrict__ dv, size_t nq8, size_t nkv8,
                                   float scale) {
  pdl_enter();
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const float* src;
  __nv_bfloat16* dst;
  float mul;
  if (i < nq8) {
    src = dq_acc; dst = dq; mul = scale;
  } else if ((i -= nq8) < nkv8) {
    src = dk_acc; dst = dk; mul = scale;
  } else if ((i -= nkv8) < nkv8) {
    src = dv_acc; dst = dv; mul = 1.f;
  } else {
    return;
  }
  const float4 a = __ldcs(reinterpret_cast<const float4*>(src) + 2 * i);
  const float4 b = __ldcs(reinterpret_cast<const float4*>(src) + 2 * i + 1);
  uint4 out;
  out.x = pack_bf16x2(a.x * mul, a.y * mul);
  out.y = pack_bf16x2(a.z * mul, a.w * mul);
  out.z = pack_bf16x2(b.x * mul, b.y * mul);
  out.w = pack_bf16x2(b.z * mul, b.w * mul);
  reinterpret_cast<uint4*>(dst)[i] = out;
}

// ---------------------------------------------------------------- main kernel

__global__ void __launch_bounds__(kBwdThreads, 1)
    sparse_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_do, const int* __restrict__ lists,
                      const int* __restrict__ list_len, const int* __restrict__ order,
                      int max_items, const int32_t* __restrict__ cu,
                      const float* __restrict__ lsd, const int4* __restrict__ items,
                      const int* __restrict__ num_items, int Hq, int Hkv, float scale,
                      float* __restrict__ dq_acc, float* __restrict__ dk_acc,
                      float* __restrict__ dv_acc, int* __restrict__ item_ctr,
                      uint32_t* status) {
  pdl_enter();
  constexpr int G = 16;
  const int n_items = *num_items;
  if (static_cast<int>(blockIdx.x) >= n_items) return;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {   // the tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(status, kStatusBounds);
    return;
  }
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
  const int g = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.ld_full[i], 1);
      mbar_init(&sm.ld_empty[i], 1);
    }
    for (int z = 0; z < 2; ++z) {
      mbar_init(&sm.s_full[z], 1);
      mbar_init(&sm.dp_full[z], 1);
      mbar_init(&sm.p_full[z], kGroupThreads);
      mbar_init(&sm.ds_full[z], kGroupThreads);
      mbar_init(&sm.dv_done[z], 1);
      mbar_init(&sm.dq_full[z], 1);
      mbar_init(&sm.dq_free[z], kGroupThreads);
    }
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_free, 2 * kGroupThreads);
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(&sm.item_full[i], 1);
      mbar_init(&sm.item_empty[i], kItemReaders);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // Half-chunk u of this CTA (counted over all its items) uses stage u % 4 and
  // TMEM slot / compute warpgroup u & 1.
  if (warp == 0 || warp == kLoaderWarp1) {
    // ------------------------------------------------------------ producers
    // warp 0 loads K_b / V_b and the even half-chunks, kLoaderWarp1 the odd ones
    const uint32_t par = (warp == 0) ? 0u : 1u;
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_do);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    bool alive = true;
    uint32_t u = 0;
    int pending = 0;
    if (par == 0 && lane == 0) pending = atomicAdd(item_ctr + g, 1);
    for (int itl = 0; alive; ++itl) {
      // Items are claimed in the order bwd_lists_kernel set, first come first
      // served: warp 0 takes the next one from the KV head's counter and
      // publishes its id (-1 once none are left) in slot itl % kItemSlots, where
      // the other roles read it.
      const int si = itl % kItemSlots;
      const uint32_t sph = (itl / kItemSlots) & 1;
      int it = -1;
      if (lane == 0) {
        if (par == 0) {
          it = pending < n_items ? __ldg(order + static_cast<size_t>(g) * max_items + pending) : -1;
          alive = mbar_wait(&sm.item_empty[si], sph ^ 1, status, 23);
          if (alive) {
            sm.item_id[si] = it;
            mbar_arrive(&sm.item_full[si]);
            if (it >= 0) pending = atomicAdd(item_ctr + g, 1);   // next claim, in flight
          }
        } else {
          alive = mbar_wait(&sm.item_full[si], sph, status, 24);
          if (alive) {
            it = sm.item_id[si];
            mbar_arrive(&sm.item_empty[si]);
          }
        }
      }
      alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
      it = __shfl_sync(0xffffffffu, it, 0);
      if (!alive || it < 0) break;
      const int4 item = items[it];
      const int s = item.x, b = item.y;
      const int seq0 = cu[s];
      const size_t li = static_cast<size_t>(it) * Hkv + g;
      const int nlist = list_len[li];
      // lane L holds list entries 8L .. 8L+7 (half-chunks 2L and 2L+1)
      int ent[8];
      {
        const int4* src = reinterpret_cast<const int4*>(lists + li * kBwdSegment) + 2 * lane;
        int4 e0 = make_int4(0, 0, 0, 0), e1 = e0;
        if (8 * lane < nlist) {
          e0 = __ldg(src);
          e1 = __ldg(src + 1);
        }
        ent[0] = e0.x; ent[1] = e0.y; ent[2] = e0.z; ent[3] = e0.w;
        ent[4] = e1.x; ent[5] = e1.y; ent[6] = e1.z; ent[7] = e1.w;
      }
      if (lane == 0 && par == 0) {
        alive = mbar_wait(&sm.kv_empty, (itl & 1) ^ 1, status, 21);
        if (alive) {
          mbar_arrive_expect_tx(&sm.kv_full, 2 * kTile);
          const int row = seq0 + b * kBlock;
          tma_load_3d(sm.k, &tm_k, &sm.kv_full, 0, g, row);
          tma_load_3d(sm.k + kHalf, &tm_k, &sm.kv_full, 64, g, row);
          tma_load_3d(sm.v, &tm_v, &sm.kv_full, 0, g, row);
          tma_load_3d(sm.v + kHalf, &tm_v, &sm.kv_full, 64, g, row);
        }
      }
      alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
      const int nh = (nlist + kHcTok - 1) / kHcTok;
      for (int j = 0; alive && j < nh; ++j, ++u) {
        if ((u & 1u) != par) continue;
        const int n = min(kHcTok, nlist - kHcTok * j);
        const int st = u % kStages;
        if (lane == 0)
          alive = mbar_wait(&sm.ld_empty[st], ((u / kStages) & 1) ^ 1, status, 22);
        alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
        if (!alive) break;
        // positions of the half-chunk's tokens (slots >= n repeat slot 0)
        int pos = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int pe = __shfl_sync(0xffffffffu, ent[e], (j >> 1) & 31);
          if (lane == e - 4 * (j & 1)) pos = pe;
        }
        const int pos0 = __shfl_sync(0xffffffffu, pos, 0);
        if (lane < kHcTok) sm.tok[st][lane] = (lane < n) ? pos : -1;
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&sm.ld_full[st], kStageBytes + kHcTok * G * 8);
        __syncwarp();
        if (lane < kHcTok) {
          // one 4 KB box per token and tensor: rows (head octet, D half, head % 8)
          const int t = seq0 + ((lane < n) ? pos : pos0);
          uint8_t* qb = sm.stage[st] + lane * kTokBytes;
          tma_load_5d(qb, &tm_q, &sm.ld_full[st], 0, 0, 0, 2 * g, t);
          tma_load_5d(qb + kStageBytes / 2, &tm_do, &sm.ld_full[st], 0, 0, 0, 2 * g, t);
          bulk_load(&sm.lsd[st][lane * 2 * G], lsd + (static_cast<size_t>(t) * Hq + g * G) * 2, G * 8,
                    &sm.ld_full[st]);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      const uint32_t ka = smem_u32(sm.k), va = smem_u32(sm.v);
      uint32_t u0 = 0;
      bool ok = true;
      int ii = 0;      // items with work
      for (int itl = 0;; ++itl) {
        const int si = itl % kItemSlots;
        if (!(ok = mbar_wait(&sm.item_full[si], (itl / kItemSlots) & 1, status, 38))) break;
        const int it = sm.item_id[si];
        mbar_arrive(&sm.item_empty[si]);
        if (it < 0) break;
        const int nlist = list_len[static_cast<size_t>(it) * Hkv + g];
        const int nh = (nlist + kHcTok - 1) / kHcTok;
        if (!(ok = mbar_wait(&sm.kv_full, itl & 1, status, 31))) break;
        tc_fence_after();
        for (int j = 0; ok && j <= nh; ++j) {
          if (j < nh) {
            // S^T and dP^T of half-chunk u into slot z
            const uint32_t u = u0 + j;
            const int z = u & 1, st = u % kStages;
            const uint32_t slot = tmem + kColSlot + 128 * z;
            if (!(ok = mbar_wait(&sm.ld_full[st], (u / kStages) & 1, status, 32))) break;
            if (u >= 2 && !(ok = mbar_wait(&sm.dv_done[z], ((u - 2) >> 1) & 1, status, 33))) break;
            tc_fence_after();
            const uint32_t qa = smem_u32(sm.stage[st]), da = qa + kStageBytes / 2;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t ao = (kk >> 2) * kHalf + (kk & 3) * 32;
              const uint32_t bo = (kk >> 2) * 1024 + (kk & 3) * 32;
              umma_bf16(slot, sdesc_sw128(ka + ao, 16, 1024), sdesc_sw128(qa + bo, 16, 2048),
                        kIdescS, kk > 0);
            }
            umma_commit(&sm.s_full[z]);
            if (u >= 2 && !(ok = mbar_wait(&sm.dq_free[z], ((u - 2) >> 1) & 1, status, 34))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t ao = (kk >> 2) * kHalf + (kk & 3) * 32;
              const uint32_t bo = (kk >> 2) * 1024 + (kk & 3) * 32;
              umma_bf16(slot + kHc, sdesc_sw128(va + ao, 16, 1024), sdesc_sw128(da + bo, 16, 2048),
                        kIdescS, kk > 0);
            }
            umma_commit(&sm.dp_full[z]);
          }
          if (j >= 1) {
            // dV, dK and dQ^T of half-chunk v = u - 1
            const uint32_t v = u0 + j - 1;
            const int z = v & 1, st = v % kStages;
            const uint32_t slot = tmem + kColSlot + 128 * z;
            const uint32_t qa = smem_u32(sm.stage[st]), da = qa + kStageBytes / 2;
            const uint32_t sa = smem_u32(sm.dst[z]);
            const bool first = (j == 1);
            if (first && ii > 0 && !(ok = mbar_wait(&sm.acc_free, (ii - 1) & 1, status, 35))) break;
            if (!(ok = mbar_wait(&sm.p_full[z], (v >> 1) & 1, status, 36))) break;
            tc_fence_after();
            // dV += P^T dO (P^T packed in the slot's first 32 columns; dO read
            // MN-major: one token = 16 K-rows per step)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_tmem_a(tmem + kColDV, slot + kk * 8,
                               sdesc_sw128(da + kk * kTokBytes, 1024, 2048), kIdescKM,
                               !(first && kk == 0));
            umma_commit(&sm.dv_done[z]);
            if (!(ok = mbar_wait(&sm.ds_full[z], (v >> 1) & 1, status, 37))) break;
            tc_fence_after();
            // dK += dS^T Q
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(tmem + kColDK, sdesc_sw128(sa + kk * 32, 16, 1024),
                        sdesc_sw128(qa + kk * kTokBytes, 1024, 2048), kIdescKM,
                        !(first && kk == 0));
            umma_commit(&sm.ld_empty[st]);   // Q / dO of the stage consumed
            // dQ^T = K^T dS^T  (M = head dim, N = the 64 columns) into the dP^T columns
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16(slot + kHc, sdesc_sw128(ka + kk * 2048, kHalf, 1024),
                        sdesc_sw128(sa + kk * 2048, kHalf, 1024), kIdescQ, kk > 0);
            umma_commit(&sm.dq_full[z]);
          }
        }
        if (!ok) break;
        if (nh > 0) {
          umma_commit(&sm.acc_full);   // dK, dV of this item are final
          ++ii;
        }
        umma_commit(&sm.kv_empty);     // K_b / V_b free once this item's MMAs are done
        u0 += nh;
      }
    }
  } else {
    // ------------------------------------------------------------ compute
    const int cw = warp - 2;                // 0..7
    const int z = cw >> 2;                  // warpgroup = TMEM slot: half-chunks u with u & 1 == z
    const int subp = warp & 3;              // TMEM sub-partition (lanes 32 subp ..)
    const int r = subp * 32 + lane;         // key row; also the head-dim row of dQ^T
    const uint32_t trow = static_cast<uint32_t>(subp * 32) << 16;
    const uint32_t slot = tmem + kColSlot + 128 * z + trow;
    const float sl2 = scale * kLog2e;
    uint32_t u0 = 0;
    int ii = 0;
    bool ok = true;
    for (int itl = 0;; ++itl) {
      const int si = itl % kItemSlots;
      if (!(ok = __all_sync(0xffffffffu,
                            mbar_wait(&sm.item_full[si], (itl / kItemSlots) & 1, status, 40))))
        break;
      const int it = sm.item_id[si];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.item_empty[si]);
      if (it < 0) break;
      const int4 item = items[it];
      const int s = item.x, b = item.y;
      const int seq0 = cu[s];
      const int len = cu[s + 1] - seq0;
      const int kp = b * kBlock + r;        // key position of this row
      const int nlist = list_len[static_cast<size_t>(it) * Hkv + g];
      const int nh = (nlist + kHcTok - 1) / kHcTok;
      for (int j = 0; j < nh; ++j) {
        const uint32_t u = u0 + j;
        if ((u & 1) != static_cast<uint32_t>(z)) continue;
        const int st = u % kStages;
        const uint32_t ph = (u >> 1) & 1;
        if (!(ok = mbar_wait(&sm.ld_full[st], (u / kStages) & 1, status, 41))) break;
        int tokp[kHcTok];
#pragma unroll
        for (int i = 0; i < kHcTok; ++i) tokp[i] = sm.tok[st][i];
        const float* ls = sm.lsd[st];

        // ---- P^T = exp2(S^T * scale log2e - lse log2e), causally masked
        if (!(ok = mbar_wait(&sm.s_full[z], ph, status, 42))) break;
        __syncwarp();
        tc_fence_after();
        float p[kHc];
        {
          uint32_t sv[kHc];
          tmem_ld32(slot, sv);
          tmem_ld32(slot + 32, sv + 32);
          tmem_ld_wait();
          const float2 sl2v = make_float2(sl2, sl2);
#pragma unroll
          for (int c4 = 0; c4 < kHc / 4; ++c4) {   // columns 4 c4 .. 4 c4 + 3 of token c4 / 4
            const float4 nl = *reinterpret_cast<const float4*>(ls + 32 * (c4 >> 2) + 4 * (c4 & 3));
            const float2 y0 = ffma2(make_float2(__uint_as_float(sv[4 * c4]), __uint_as_float(sv[4 * c4 + 1])),
                                    sl2v, make_float2(nl.x, nl.y));
            const float2 y1 = ffma2(make_float2(__uint_as_float(sv[4 * c4 + 2]), __uint_as_float(sv[4 * c4 + 3])),
                                    sl2v, make_float2(nl.z, nl.w));
            p[4 * c4] = ex2(y0.x);
            p[4 * c4 + 1] = ex2(y0.y);
            p[4 * c4 + 2] = ex2(y1.x);
            p[4 * c4 + 3] = ex2(y1.y);
          }
          // causal mask (keys after the query: only in the token's own block)
          // and padding slots (token -1)
          bool mask[kHcTok];
          bool any = false;
#pragma unroll
          for (int i = 0; i < kHcTok; ++i) {
            mask[i] = kp > tokp[i];
            any |= mask[i];
          }
          if (__any_sync(0xffffffffu, any)) {
#pragma unroll
            for (int c = 0; c < kHc; ++c) p[c] = mask[c >> 4] ? 0.f : p[c];
          }
          uint32_t pk[kHc / 2];
#pragma unroll
          for (int c = 0; c < kHc / 2; ++c) pk[c] = pack_bf16x2(p[2 * c], p[2 * c + 1]);
          tmem_st16(slot, pk);
          tmem_st16(slot + 16, pk + 16);
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&sm.p_full[z]);
        // -Delta of the 64 columns, fetched while dP^T is computed (the dS step
        // below then reads P^T back from TMEM and needs no shared-memory loads)
        float4 ndl[kHc / 4];
#pragma unroll
        for (int q4 = 0; q4 < kHc / 4; ++q4)
          ndl[q4] = *reinterpret_cast<const float4*>(ls + 32 * (q4 >> 2) + 16 + 4 * (q4 & 3));

        // ---- dS^T = P^T (dP^T - Delta) -> shared memory (K-major, rows = keys)
        if (!(ok = mbar_wait(&sm.dp_full[z], ph, status, 43))) break;
        __syncwarp();
        tc_fence_after();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t dv[32], pb[16];
          tmem_ld32(slot + kHc + 32 * hf, dv);
          tmem_ld16(slot + 16 * hf, pb);       // P^T of these 32 columns, bf16 pairs
          tmem_ld_wait();
#pragma unroll
          for (int c = 4 * hf; c < 4 * hf + 4; ++c) {
            float x[8];
#pragma unroll
            for (int e4 = 0; e4 < 2; ++e4) {
              const int c0 = 8 * c + 4 * e4;   // token c0 / 16, heads c0 % 16 ..
              const int d0 = c0 - 32 * hf;
              const float4 nd = ndl[c0 / 4];
              const float2 t0 = fadd2(make_float2(__uint_as_float(dv[d0]), __uint_as_float(dv[d0 + 1])),
                                      make_float2(nd.x, nd.y));
              const float2 t1 = fadd2(make_float2(__uint_as_float(dv[d0 + 2]), __uint_as_float(dv[d0 + 3])),
                                      make_float2(nd.z, nd.w));
              const float2 p01 = unpack_bf16x2(pb[d0 / 2]), p23 = unpack_bf16x2(pb[d0 / 2 + 1]);
              const float2 x0 = fmul2(p01, t0);
              const float2 x1 = fmul2(p23, t1);
              x[4 * e4] = x0.x;
              x[4 * e4 + 1] = x0.y;
              x[4 * e4 + 2] = x1.x;
              x[4 * e4 + 3] = x1.y;
            }
            uint4 pk;
            pk.x = pack_bf16x2(x[0], x[1]);
            pk.y = pack_bf16x2(x[2], x[3]);
            pk.z = pack_bf16x2(x[4], x[5]);
            pk.w = pack_bf16x2(x[6], x[7]);
            *reinterpret_cast<uint4*>(sm.dst[z] + sw128_offset(r, c)) = pk;
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&sm.ds_full[z]);

        // ---- dQ^T (lane = head-dim row r, 64 columns) added into the fp32
        // accumulator: per column a warp adds 32 consecutive floats of one row
        if (!(ok = mbar_wait(&sm.dq_full[z], ph, status, 45))) break;
        __syncwarp();
        tc_fence_after();
        {
          uint32_t qv[kHc];
          tmem_ld32(slot + kHc, qv);
          tmem_ld32(slot + kHc + 32, qv + 32);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&sm.dq_free[z]);          // the TMEM columns are free once read
#pragma unroll
          for (int ti = 0; ti < kHcTok; ++ti) {
            if (tokp[ti] < 0) continue;
            float* row = dq_acc + (static_cast<size_t>(seq0 + tokp[ti]) * Hq + g * G) * kD + r;
#pragma unroll
            for (int hd = 0; hd < G; ++hd) red_add_f32(row + hd * kD, __uint_as_float(qv[16 * ti + hd]));
          }
        }
      }
      if (!ok) break;
      u0 += nh;
      if (nh == 0) continue;
      // ---- dK (warpgroup 0) or dV (warpgroup 1) of this item -> fp32 accumulator
      if (!(ok = mbar_wait(&sm.acc_full, ii & 1, status, 46))) break;
      __syncwarp();
      tc_fence_after();
      {
        const bool key_valid = kp < len;
        float* dst_acc = (z == 0) ? dk_acc : dv_acc;
        const uint32_t col = (z == 0) ? kColDK : kColDV;
        float4* dst = reinterpret_cast<float4*>(
            dst_acc + (static_cast<size_t>(seq0 + kp) * Hkv + g) * kD);
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t a[32];
          tmem_ld32(tmem + col + trow + c0, a);
          tmem_ld_wait();
          if (key_valid) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              atomicAdd(dst + c0 / 4 + q,
                        make_float4(__uint_as_float(a[4 * q]), __uint_as_float(a[4 * q + 1]),
                                    __uint_as_float(a[4 * q + 2]), __uint_as_float(a[4 * q + 3])));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.acc_free);
      ++ii;
    }
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- host

static int bwd_windows(int max_seqlen) { return (max_seqlen + kBwdSegment - 1) / kBwdSegment; }

static int bwd_max_items(int T, int S, int max_seqlen) {
  // items of sequence s <= (windows of s) x (blocks of s) <= (T / W + S) x max_nb
  const long long max_nb = (max_seqlen + kBlock - 1) / kBlock;
  const long long n = (static_cast<long long>(T) / kBwdSegment + S) * max_nb;
  return static_cast<int>(n < (1LL << 30) ? n : (1LL << 30));
}

msa_status_t launch_bwd_clear(const BwdWorkspace& ws, int Hkv, cudaStream_t stream) {
  // the three accumulators and the item counters are carved back to back: one
  // clear covers them
  const size_t acc_bytes = reinterpret_cast<uint8_t*>(ws.item_ctr + Hkv) -
                           reinterpret_cast<uint8_t*>(ws.dq_acc);
  if (cudaMemsetAsync(ws.dq_acc, 0, acc_bytes, stream) != cudaSuccess)
    return fail(MSA_ERR_CUDA, "workspace clear failed");
  return MSA_OK;
}

BwdWorkspace carve_bwd_workspace(WsCursor& ws, int T, int S, int Hq, int Hkv, int max_seqlen) {
  BwdWorkspace w;
  w.max_items = bwd_max_items(T, S, max_seqlen);
  w.items = ws.take<int4>(w.max_items);
  w.num_items = ws.take<int>(1);
  w.lists = ws.take<int>(static_cast<size_t>(w.max_items) * Hkv * kBwdSegment);
  w.list_len = ws.take<int>(static_cast<size_t>(w.max_items) * Hkv);
  w.order = ws.take<int>(static_cast<size_t>(w.max_items) * Hkv);
  w.lists_done = ws.take<int>(Hkv);
  w.lsd = ws.take<float>(static_cast<size_t>(T) * Hq * 2);
  // the three accumulators and the item counters stay adjacent and in this
  // order: one clear covers them
  w.dq_acc = ws.take<float>(static_cast<size_t>(T) * Hq * kD);
  w.dk_acc = ws.take<float>(static_cast<size_t>(T) * Hkv * kD);
  w.dv_acc = ws.take<float>(static_cast<size_t>(T) * Hkv * kD);
  w.item_ctr = ws.take<int>(Hkv);
  return w;
}

msa_status_t launch_sparse_bwd(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, const int32_t* sel,
                               const int32_t* cu, int S, int T, int Hq, int Hkv, int max_seqlen,
                               float scale, const BwdWorkspace& ws, void* dq, void* dk, void* dv,
                               bool clear_acc, cudaStream_t stream) {
  const int G = Hq / Hkv;
  if (G != 16)
    return fail(MSA_ERR_UNSUPPORTED, "backward supports Hq/Hkv = 16 (got %d)", G);
  CUtensorMap tq, tk, tv, tdo;
  // Q / dO as (d % 64, head % 8, d / 64, head / 8, token): a (64, 8, 2, 2, 1)
  // box is one token's 16 heads of KV group g in the order the kernel reads.
  const uint64_t dq5[5] = {64, 8, 2, static_cast<uint64_t>(Hq / 8), static_cast<uint64_t>(T)};
  const uint64_t sq5[4] = {static_cast<uint64_t>(kD) * 2, 128, 8 * static_cast<uint64_t>(kD) * 2,
                           static_cast<uint64_t>(Hq) * kD * 2};
  const uint32_t bq5[5] = {64, 8, 2, 2, 1};
  const uint64_t dkv3[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hkv),
                            static_cast<uint64_t>(T)};
  const uint32_t bkv[3] = {64, 1, 128};
  if (!make_tmap_bf16_strided(&tq, q, 5, dq5, sq5, bq5) ||
      !make_tmap_bf16_strided(&tdo, dout, 5, dq5, sq5, bq5) ||
      !make_tmap_bf16(&tk, k, 3, dkv3, bkv) || !make_tmap_bf16(&tv, v, 3, dkv3, bkv))
    return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the backward");
  uint32_t* st = nullptr;
  if (msa_status_t e_ = status_word(&st); e_ != MSA_OK) return e_;

  const size_t nq = static_cast<size_t>(T) * Hq * kD;
  const size_t nkv = static_cast<size_t>(T) * Hkv * kD;
  if (clear_acc) {
    const msa_status_t e = launch_bwd_clear(ws, Hkv, stream);
    if (e != MSA_OK) return e;
  }

  const size_t rows = static_cast<size_t>(T) * Hq;
  {
    // CTA 0 also lists the work items and clears the lists kernel's counters
    TraceScope trace_("bwd_delta_kernel", stream);
    const size_t per_block = 256 / 16 * kDeltaRows;
    launch_pdl(bwd_delta_kernel, static_cast<unsigned>((rows + per_block - 1) / per_block), 256,
        0, stream,
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, ws.lsd,
        rows, cu, S, max_seqlen, bwd_windows(max_seqlen), ws.items, ws.num_items, ws.max_items,
        ws.lists_done, Hkv, st);
  }
  {
    // the last CTA of each KV head also writes that head's claim order
    // measured on GB300: a 16k pack (134 MB of fp32 dQ) runs 2 % faster with
    // its last third sorted (every item sorted: as fast, but 1.7x the DRAM
    // bytes); a 32k pack with 64 heads (1 GB) 1.7 % slower (13 % fully sorted)
    const int tail_div = nq * sizeof(float) <= 2 * device_l2_bytes() ? 3 : 5;
    const int sms = device_sm_count();
    dim3 lgrid(static_cast<unsigned>(ws.max_items < 4 * sms ? ws.max_items : 4 * sms), Hkv);
    TraceScope trace_("bwd_lists_kernel", stream);
    launch_pdl(bwd_lists_kernel, lgrid, kBwdSegment, 0, stream, cu, sel, ws.items, ws.num_items,
        Hkv, ws.lists, ws.list_len, ws.lists_done, ws.max_items, ws.order, tail_div);
  }
  msa_status_t e = check_launch("bwd_delta/lists");
  if (e != MSA_OK) return e;

  const size_t smem = sizeof(BwdSmem);
  {
    const msa_status_t e = ensure_smem(sparse_bwd_kernel, smem, "sparse_bwd_kernel");
    if (e != MSA_OK) return e;
  }
  const int per_head = (device_sm_count() + Hkv - 1) / Hkv;
  dim3 grid(static_cast<unsigned>(per_head < ws.max_items ? per_head : ws.max_items), Hkv);
  {
    TraceScope trace_("sparse_bwd_kernel", stream);
    launch_pdl(sparse_bwd_kernel, grid, kBwdThreads, smem, stream,
        tq, tk, tv, tdo, ws.lists, ws.list_len, ws.order, ws.max_items, cu, ws.lsd, ws.items, ws.num_items, Hq, Hkv, scale,
        ws.dq_acc, ws.dk_acc, ws.dv_acc, ws.item_ctr, st);
  }
  e = check_launch("sparse_bwd_kernel");
  if (e != MSA_OK) return e;

  {
    const size_t n8 = nq / 8 + 2 * (nkv / 8);
    TraceScope trace_("bwd_convert_kernel", stream);
    launch_pdl(bwd_convert_kernel, static_cast<unsigned>((n8 + 255) / 256), 256, 0, stream,
        ws.dq_acc, ws.dk_acc, ws.dv_acc, static_cast<__nv_bfloat16*>(dq),
        static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), nq / 8, nkv / 8, scale);
  }
  return check_launch("bwd_convert_kernel");
}

}  // namespace msa
