// Block-sparse attention backward ("#4581", "Kernel tuning": dQ and dK/dV of
// the block-sparse kernel; "MiniMax-M3.1-Flash", 5.4 "Notable quirks": the
// indexer is frozen, so the selection is a constant here).
//
// KV-major schedule.  A work item is (KV head g, key block b of sequence s, a
// 256-position window of candidate query positions).  Items are listed window
// by window, so the items running at any moment add into dQ rows of a few
// windows only and the fp32 dQ accumulator lines stay in L2.  Persistent CTAs
// (one per SM) stride over the items.  Per item the CTA holds K_b and V_b in
// shared memory and streams the query tokens of the window that selected b, in
// ascending order, in chunks of 128/G tokens x G heads = 128 columns.  A
// pre-pass (bwd_lists_kernel) lists, per item, the window's tokens that
// selected the block (one thread per candidate, ballot compaction).
//   producer (warp 0): loads the chunk's Q and dO rows by TMA (one box per
//            token) and its lse / Delta by bulk copies into a 2-stage ring
//   MMA (warp 1): S^T = K_b Q^T -> TMEM, dP^T = V_b dO^T -> TMEM,
//            dV += P^T dO (P^T read from TMEM), dK += dS^T Q,
//            dQ = dS K_b (dS^T in shared memory read as an MN-major operand)
//   compute (warps 2..9, thread = key row x 64 columns):
//            P^T = exp2(S^T scale log2e - lse log2e), causally masked, packed
//            to bf16 into TMEM; dS^T = P^T (dP^T - Delta) to shared memory;
//            then dQ rows (lane = column) are staged, 128B-swizzled, in the
//            chunk's own Q/dO buffers, which the producer adds into the fp32
//            accumulator with TMA reduce-add before refilling the stage; at the
//            end of an item dK and dV go to their accumulators with atomics.
// A last kernel scales and converts the accumulators to bf16.
#include "kernels.cuh"

namespace msa {

namespace {

constexpr int kBwdThreads = 320;            // warp 0 TMA, warp 1 MMA, warps 2..9 compute
constexpr int kComputeThreads = 256;
constexpr int kTile = 128 * 128 * 2;
constexpr int kHalf = kTile / 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kIdescKK = idesc_bf16(128, 128, false, false);   // both K-major
constexpr uint32_t kIdescKM = idesc_bf16(128, 128, false, true);    // B MN-major
constexpr uint32_t kIdescMM = idesc_bf16(128, 128, true, true);     // both MN-major
// TMEM columns
constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 384;

struct BwdSmem {
  uint8_t k[kTile];
  uint8_t v[kTile];
  uint8_t q[2][kTile];
  uint8_t dout[2][kTile];
  uint8_t dst[kTile];
  float lse[2][128];      // natural-log lse of the chunk's 128 columns (bulk-copied)
  float delta[2][128];
  int tok[2][16];
  int ntok[2];
  uint64_t kv_full, kv_empty;
  uint64_t ld_full[2], ld_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full, dv_done, dq_full, dq_free;
  uint32_t tmem_base;
};
static_assert(sizeof(BwdSmem) <= 232448, "backward shared memory above the 227 KB limit");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// One CTA.  Pairs (window w, sequence s) in w-major order; pair (w, s) holds the
// key blocks b that some query of window w can select: 128 b < min(len, (w+1) W).
// Each becomes an item (s, b, first position, end position) of that window.
__global__ void __launch_bounds__(1024) bwd_items_kernel(const int32_t* __restrict__ cu, int S,
                                                         int num_windows,
                                                         int4* __restrict__ items,
                                                         int* __restrict__ num_items,
                                                         int max_items, uint32_t* status) {
  __shared__ int warp_sums[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const long long npairs = static_cast<long long>(num_windows) * S;
  for (long long base = 0; base < npairs; base += blockDim.x) {
    const long long pi = base + threadIdx.x;
    int s = 0, w = 0, len = 0, cnt = 0;
    if (pi < npairs) {
      w = static_cast<int>(pi / S);
      s = static_cast<int>(pi % S);
      len = cu[s + 1] - cu[s];
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

// One CTA of kBwdSegment threads per (item, KV head), grid-striding over items:
// thread t checks candidate position first + t; the matches are compacted in
// ascending order into the item's list.
__global__ void __launch_bounds__(kBwdSegment) bwd_lists_kernel(
    const int32_t* __restrict__ cu, const int32_t* __restrict__ sel,
    const int4* __restrict__ items, const int* __restrict__ num_items, int Hkv,
    int* __restrict__ lists, int* __restrict__ list_len) {
  static_assert(kBwdSegment == 256, "one thread per candidate position");
  __shared__ int warp_cnt[kBwdSegment / 32];
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
}

// ---------------------------------------------------------------- Delta

// delta[t, i] = sum_d dout[t, i, d] * o[t, i, d]; one warp per row.
__global__ void bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                 const __nv_bfloat16* __restrict__ dout, float* __restrict__ delta,
                                 size_t rows) {
  const size_t row = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint2 a = reinterpret_cast<const uint2*>(o + row * kD)[lane];
  const uint2 b = reinterpret_cast<const uint2*>(dout + row * kD)[lane];
  const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float2 x = __bfloat1622float2(a2[j]);
    const float2 y = __bfloat1622float2(b2[j]);
    acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (lane == 0) delta[row] = acc;
}

// ---------------------------------------------------------------- convert

__global__ void bwd_convert_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst,
                                   size_t n8, float mul) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(src)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(src)[2 * i + 1];
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
                      const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_dq, const int* __restrict__ lists,
                      const int* __restrict__ list_len, const int32_t* __restrict__ cu,
                      const float* __restrict__ lse,
                      const float* __restrict__ delta, const int4* __restrict__ items,
                      const int* __restrict__ num_items, int Hq, int Hkv, float scale,
                      float* __restrict__ dq_acc, float* __restrict__ dk_acc,
                      float* __restrict__ dv_acc, uint32_t* status) {
  constexpr int G = 16, tpt = 8;    // heads per KV group, tokens per chunk
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.ld_full[i], 1);
      mbar_init(&sm.ld_empty[i], 1 + kComputeThreads);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.dp_full, 1);
    mbar_init(&sm.p_full, kComputeThreads);
    mbar_init(&sm.ds_full, kComputeThreads);
    mbar_init(&sm.dv_done, 1);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_free, kComputeThreads);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_do);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    uint32_t cg = 0;
    bool alive = true;
    int itl = 0;
    // dQ rows of the chunk that last used a stage are staged in that stage's Q/dO
    // buffers (8 tokens x 4 boxes of 16 heads x 32 fp32, 128B-swizzled); before the
    // stage is refilled they are added into the fp32 accumulator by TMA reduce.
    int pend_n[2] = {0, 0}, pend_seq0[2] = {0, 0};
    auto flush_dq = [&](int st) {
      if (pend_n[st] == 0) return;
      if (lane < pend_n[st]) {
        const int y = (pend_seq0[st] + sm.tok[st][lane]) * Hq + g * G;
        const uint8_t* box = (lane < 4 ? sm.q[st] : sm.dout[st]) + (lane & 3) * 4 * 2048;
#pragma unroll
        for (int j = 0; j < 4; ++j) tma_reduce_add_2d(&tm_dq, box + j * 2048, 32 * j, y);
        bulk_commit_group();
        bulk_wait_read_all();
      }
      __syncwarp();
      pend_n[st] = 0;
    };
    for (int it = blockIdx.x; alive && it < n_items; it += gridDim.x, ++itl) {
      const int4 item = items[it];
      const int s = item.x, b = item.y;
      const int seq0 = cu[s];
      const size_t li = static_cast<size_t>(it) * Hkv + g;
      const int nlist = list_len[li];
      // lane L holds list entries 8L .. 8L+7 (chunk L)
      int ent[tpt];
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
      if (lane == 0) {
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
      const int nchunks = (nlist + tpt - 1) / tpt;
      for (int c = 0; alive && c <= nchunks; ++c) {
        const int n = (c < nchunks) ? min(tpt, nlist - tpt * c) : 0;   // 0: end of the item
        const int st = cg & 1;
        if (lane == 0) alive = mbar_wait(&sm.ld_empty[st], ((cg >> 1) & 1) ^ 1, status, 22);
        alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
        if (!alive) break;
        flush_dq(st);
        // positions of the chunk's tokens, broadcast from lane c (slots >= n repeat slot 0)
        int pos = 0;
#pragma unroll
        for (int j = 0; j < tpt; ++j) {
          const int pj = __shfl_sync(0xffffffffu, ent[j], c & 31);
          if (lane == j) pos = pj;
        }
        const int pos0 = __shfl_sync(0xffffffffu, pos, 0);
        if (lane < tpt) sm.tok[st][lane] = (lane < n) ? pos : -1;
        if (lane == 0) {
          sm.ntok[st] = n;
          if (n > 0) mbar_arrive_expect_tx(&sm.ld_full[st], 2 * kTile + tpt * 2 * G * 4);
        }
        __syncwarp();
        if (n > 0) {
          if (lane < tpt) {
            const int t = seq0 + ((lane < n) ? pos : pos0);
            const uint32_t off = lane * G * 128;
            tma_load_3d(sm.q[st] + off, &tm_q, &sm.ld_full[st], 0, g * G, t);
            tma_load_3d(sm.q[st] + kHalf + off, &tm_q, &sm.ld_full[st], 64, g * G, t);
            tma_load_3d(sm.dout[st] + off, &tm_do, &sm.ld_full[st], 0, g * G, t);
            tma_load_3d(sm.dout[st] + kHalf + off, &tm_do, &sm.ld_full[st], 64, g * G, t);
            const size_t row = static_cast<size_t>(t) * Hq + g * G;
            bulk_load(&sm.lse[st][lane * G], lse + row, G * 4, &sm.ld_full[st]);
            bulk_load(&sm.delta[st][lane * G], delta + row, G * 4, &sm.ld_full[st]);
          }
        } else if (lane == 0) {
          mbar_arrive(&sm.ld_full[st]);   // end of the item: no data
        }
        pend_n[st] = n;
        pend_seq0[st] = seq0;
        ++cg;
      }
    }
    // the last two stage uses may still hold staged dQ rows
    for (int k = 0; alive && k < 2; ++k) {
      const int st = cg & 1;
      if (pend_n[st] > 0) {
        if (lane == 0) alive = mbar_wait(&sm.ld_empty[st], ((cg >> 1) & 1) ^ 1, status, 23);
        alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
        if (alive) flush_dq(st);
      }
      ++cg;
    }
    bulk_wait_all();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      const uint32_t ka = smem_u32(sm.k), va = smem_u32(sm.v), sa = smem_u32(sm.dst);
      uint32_t cg = 0, cm = 0;
      bool ok = true;
      int itl = 0;
      for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, ++itl) {
        if (!(ok = mbar_wait(&sm.kv_full, itl & 1, status, 31))) break;
        bool first = true;
        while (ok) {
          const int st = cg & 1;
          ok = mbar_wait(&sm.ld_full[st], (cg >> 1) & 1, status, 32);
          ++cg;
          if (!ok) break;
          if (sm.ntok[st] == 0) {
            mbar_arrive(&sm.ld_empty[st]);
            break;
          }
          tc_fence_after();
          const uint32_t qa = smem_u32(sm.q[st]), da = smem_u32(sm.dout[st]);
          // S^T = K Q^T (needs P^T of the previous chunk consumed by its dV)
          if (cm > 0 && !(ok = mbar_wait(&sm.dv_done, (cm - 1) & 1, status, 33))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            umma_bf16(tmem + kColS, sdesc_sw128(ka + off, 16, 1024),
                      sdesc_sw128(qa + off, 16, 1024), kIdescKK, kk > 0);
          }
          umma_commit(&sm.s_full);
          // dP^T = V dO^T (needs dQ of the previous chunk drained)
          if (cm > 0 && !(ok = mbar_wait(&sm.dq_free, (cm - 1) & 1, status, 34))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            umma_bf16(tmem + kColDP, sdesc_sw128(va + off, 16, 1024),
                      sdesc_sw128(da + off, 16, 1024), kIdescKK, kk > 0);
          }
          umma_commit(&sm.dp_full);
          // dV += P^T dO, P^T packed in TMEM: chunk columns [64h, 64h+64) at
          // TMEM kColS + 64h .. + 32
          if (!(ok = mbar_wait(&sm.p_full, cm & 1, status, 35))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t a_t = tmem + kColS + (kk >> 2) * 64 + (kk & 3) * 8;
            umma_bf16_tmem_a(tmem + kColDV, a_t, sdesc_sw128(da + kk * 2048, kHalf, 1024),
                             kIdescKM, (!first || kk > 0));
          }
          umma_commit(&sm.dv_done);
          // dK += dS^T Q and dQ = dS K
          if (!(ok = mbar_wait(&sm.ds_full, cm & 1, status, 38))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t aoff = (kk >> 2) * kHalf + (kk & 3) * 32;
            umma_bf16(tmem + kColDK, sdesc_sw128(sa + aoff, 16, 1024),
                      sdesc_sw128(qa + kk * 2048, kHalf, 1024), kIdescKM, (!first || kk > 0));
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = kk * 2048;
            umma_bf16(tmem + kColDP, sdesc_sw128(sa + off, kHalf, 1024),
                      sdesc_sw128(ka + off, kHalf, 1024), kIdescMM, kk > 0);
          }
          umma_commit(&sm.dq_full);
          umma_commit(&sm.ld_empty[st]);
          first = false;
          ++cm;
        }
        umma_commit(&sm.kv_empty);   // K_b / V_b free once this item's MMAs are done
      }
    }
  } else {
    // ------------------------------------------------------------ compute
    const int cw = warp - 2;                // 0..7
    const int subp = warp & 3;              // TMEM sub-partition (lanes 32 subp ..)
    const int h = cw >> 2;                  // column half: chunk columns [64h, 64h + 64)
    const int r = subp * 32 + lane;         // key row; also the dQ column (token, head)
    const uint32_t trow = static_cast<uint32_t>(subp * 32) << 16;
    const float sl2 = scale * kLog2e;
    uint32_t cg = 0, cm = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const int4 item = items[it];
      const int s = item.x, b = item.y;
      const int seq0 = cu[s];
      const int len = cu[s + 1] - seq0;
      const int kp = b * kBlock + r;        // key position of this row
      int nch = 0;
      while (true) {
        const int st = cg & 1;
        if (!(ok = mbar_wait(&sm.ld_full[st], (cg >> 1) & 1, status, 41))) break;
        ++cg;
        const int n = sm.ntok[st];
        if (n == 0) {
          mbar_arrive(&sm.ld_empty[st]);
          break;
        }
        int tokp[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) tokp[i] = sm.tok[st][4 * h + i];
        const int tokd = sm.tok[st][r >> 4];     // token of this thread's dQ column
        const float* lsen = sm.lse[st] + 64 * h;
        const float* dlt = sm.delta[st] + 64 * h;

        // ---- P^T = exp2(S^T * scale log2e - lse log2e), causally masked
        if (!(ok = mbar_wait(&sm.s_full, cm & 1, status, 42))) break;
        __syncwarp();
        tc_fence_after();
        float p[64];
        {
          uint32_t sv[64];
          tmem_ld32(tmem + kColS + trow + 64 * h, sv);
          tmem_ld32(tmem + kColS + trow + 64 * h + 32, sv + 32);
          tmem_ld_wait();
#pragma unroll
          for (int j4 = 0; j4 < 16; ++j4) {
            const float4 l4 = reinterpret_cast<const float4*>(lsen)[j4];
            const float lv[4] = {l4.x * kLog2e, l4.y * kLog2e, l4.z * kLog2e, l4.w * kLog2e};
            const bool valid = kp <= tokp[j4 >> 2];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = 4 * j4 + e;
              p[j] = valid ? ex2(fmaf(__uint_as_float(sv[j]), sl2, -lv[e])) : 0.f;
            }
          }
          uint32_t pk[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) pk[j] = pack_bf16x2(p[2 * j], p[2 * j + 1]);
          tmem_st16(tmem + kColS + trow + 64 * h, pk);
          tmem_st16(tmem + kColS + trow + 64 * h + 16, pk + 16);
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&sm.p_full);

        // ---- dS^T = P^T (dP^T - Delta) -> shared memory (K-major rows = keys)
        if (!(ok = mbar_wait(&sm.dp_full, cm & 1, status, 43))) break;
        __syncwarp();
        tc_fence_after();
        {
          uint32_t dv[64];
          tmem_ld32(tmem + kColDP + trow + 64 * h, dv);
          tmem_ld32(tmem + kColDP + trow + 64 * h + 32, dv + 32);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 d0 = reinterpret_cast<const float4*>(dlt)[2 * c];
            const float4 d1 = reinterpret_cast<const float4*>(dlt)[2 * c + 1];
            const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              x[e] = p[8 * c + e] * (__uint_as_float(dv[8 * c + e]) - dd[e]);
            uint4 pk;
            pk.x = pack_bf16x2(x[0], x[1]);
            pk.y = pack_bf16x2(x[2], x[3]);
            pk.z = pack_bf16x2(x[4], x[5]);
            pk.w = pack_bf16x2(x[6], x[7]);
            *reinterpret_cast<uint4*>(sm.dst + h * kHalf + sw128_offset(r, c)) = pk;
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&sm.ds_full);

        // ---- dQ rows (lane = chunk column) -> staging in this stage's Q/dO
        // buffers (their operands are consumed once dQ is done); the producer
        // adds them into the accumulator with TMA reduce before refilling
        if (!(ok = mbar_wait(&sm.dq_full, cm & 1, status, 45))) break;
        __syncwarp();
        tc_fence_after();
        {
          uint32_t qv[64];
          tmem_ld32(tmem + kColDP + trow + 64 * h, qv);
          tmem_ld32(tmem + kColDP + trow + 64 * h + 32, qv + 32);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&sm.dq_free);           // the TMEM region is free once read
          if (tokd >= 0) {
            const int ti = r >> 4, hd = r & 15;
            uint8_t* box = (ti < 4 ? sm.q[st] : sm.dout[st]) + (ti & 3) * 4 * 2048 + hd * 128;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              uint8_t* bx = box + (2 * h + jj) * 2048;
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(bx + ((c ^ (hd & 7)) << 4)) =
                    make_uint4(qv[32 * jj + 4 * c], qv[32 * jj + 4 * c + 1],
                               qv[32 * jj + 4 * c + 2], qv[32 * jj + 4 * c + 3]);
            }
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&sm.ld_empty[st]);        // staged; done with the stage
        ++cm;
        ++nch;
      }
      // ---- dK, dV of this item (all its MMAs completed before the last dq_full)
      if (ok && nch > 0) {
        __syncwarp();
        const bool key_valid = kp < len;
        const size_t krow = (static_cast<size_t>(seq0 + kp) * Hkv + g) * kD + 64 * h;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          uint32_t a[64];
          const uint32_t col = (which == 0 ? kColDK : kColDV) + 64 * h;
          tmem_ld32(tmem + col + trow, a);
          tmem_ld32(tmem + col + trow + 32, a + 32);
          tmem_ld_wait();
          if (key_valid) {
            float4* dst = reinterpret_cast<float4*>((which == 0 ? dk_acc : dv_acc) + krow);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              atomicAdd(dst + j, make_float4(__uint_as_float(a[4 * j]), __uint_as_float(a[4 * j + 1]),
                                             __uint_as_float(a[4 * j + 2]),
                                             __uint_as_float(a[4 * j + 3])));
          }
        }
        tc_fence_before();
      }
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

BwdWorkspace carve_bwd_workspace(WsCursor& ws, int T, int S, int Hq, int Hkv, int max_seqlen) {
  BwdWorkspace w;
  w.plan = carve_plan(ws, T, S);
  w.max_items = bwd_max_items(T, S, max_seqlen);
  w.items = ws.take<int4>(w.max_items);
  w.num_items = ws.take<int>(1);
  w.lists = ws.take<int>(static_cast<size_t>(w.max_items) * Hkv * kBwdSegment);
  w.list_len = ws.take<int>(static_cast<size_t>(w.max_items) * Hkv);
  w.delta = ws.take<float>(static_cast<size_t>(T) * Hq);
  w.dq_acc = ws.take<float>(static_cast<size_t>(T) * Hq * kD);
  w.dk_acc = ws.take<float>(static_cast<size_t>(T) * Hkv * kD);
  w.dv_acc = ws.take<float>(static_cast<size_t>(T) * Hkv * kD);
  return w;
}

msa_status_t launch_sparse_bwd(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, const int32_t* sel,
                               const int32_t* cu, int S, int T, int Hq, int Hkv, int max_seqlen,
                               float scale, const BwdWorkspace& ws, void* dq, void* dk, void* dv,
                               cudaStream_t stream) {
  const int G = Hq / Hkv;
  if (G != 16)
    return fail(MSA_ERR_UNSUPPORTED, "backward supports Hq/Hkv = 16 (got %d)", G);
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t dq3[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hq),
                           static_cast<uint64_t>(T)};
  const uint64_t dkv3[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hkv),
                            static_cast<uint64_t>(T)};
  const uint32_t bq[3] = {64, static_cast<uint32_t>(G), 1};
  const uint32_t bkv[3] = {64, 1, 128};
  CUtensorMap tdq;
  const uint64_t dacc[2] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(T) * Hq};
  const uint32_t bacc[2] = {32, 16};
  if (!make_tmap_bf16(&tq, q, 3, dq3, bq) || !make_tmap_bf16(&tdo, dout, 3, dq3, bq) ||
      !make_tmap_bf16(&tk, k, 3, dkv3, bkv) || !make_tmap_bf16(&tv, v, 3, dkv3, bkv) ||
      !make_tmap_f32(&tdq, ws.dq_acc, 2, dacc, bacc))
    return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the backward");
  uint32_t* st = status_word();

  const size_t nq = static_cast<size_t>(T) * Hq * kD;
  const size_t nkv = static_cast<size_t>(T) * Hkv * kD;
  if (cudaMemsetAsync(ws.dq_acc, 0, nq * sizeof(float), stream) != cudaSuccess ||
      cudaMemsetAsync(ws.dk_acc, 0, nkv * sizeof(float), stream) != cudaSuccess ||
      cudaMemsetAsync(ws.dv_acc, 0, nkv * sizeof(float), stream) != cudaSuccess)
    return fail(MSA_ERR_CUDA, "workspace clear failed");

  const size_t rows = static_cast<size_t>(T) * Hq;
  {
    TraceScope trace_("bwd_delta_kernel", stream);
    bwd_delta_kernel<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), ws.delta,
        rows);
  }
  {
    TraceScope trace_("bwd_items_kernel", stream);
    bwd_items_kernel<<<1, 1024, 0, stream>>>(cu, S, bwd_windows(max_seqlen), ws.items,
                                             ws.num_items, ws.max_items, st);
  }
  {
    const int sms = device_sm_count();
    dim3 lgrid(static_cast<unsigned>(ws.max_items < 4 * sms ? ws.max_items : 4 * sms), Hkv);
    TraceScope trace_("bwd_lists_kernel", stream);
    bwd_lists_kernel<<<lgrid, kBwdSegment, 0, stream>>>(cu, sel, ws.items, ws.num_items, Hkv,
                                                         ws.lists, ws.list_len);
  }
  msa_status_t e = check_launch("bwd_delta/items/lists");
  if (e != MSA_OK) return e;

  const size_t smem = sizeof(BwdSmem);
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(sparse_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    attr_set = true;
  }
  const int per_head = (device_sm_count() + Hkv - 1) / Hkv;
  dim3 grid(static_cast<unsigned>(per_head < ws.max_items ? per_head : ws.max_items), Hkv);
  {
    TraceScope trace_("sparse_bwd_kernel", stream);
    sparse_bwd_kernel<<<grid, kBwdThreads, smem, stream>>>(
        tq, tk, tv, tdo, tdq, ws.lists, ws.list_len, cu, lse, ws.delta, ws.items, ws.num_items, Hq,
        Hkv, scale,
        ws.dq_acc, ws.dk_acc, ws.dv_acc, st);
  }
  e = check_launch("sparse_bwd_kernel");
  if (e != MSA_OK) return e;

  {
    TraceScope trace_("bwd_convert_kernel", stream);
    bwd_convert_kernel<<<static_cast<unsigned>((nq / 8 + 255) / 256), 256, 0, stream>>>(
        ws.dq_acc, static_cast<__nv_bfloat16*>(dq), nq / 8, scale);
  }
  {
    TraceScope trace_("bwd_convert_kernel", stream);
    bwd_convert_kernel<<<static_cast<unsigned>((nkv / 8 + 255) / 256), 256, 0, stream>>>(
        ws.dk_acc, static_cast<__nv_bfloat16*>(dk), nkv / 8, scale);
  }
  {
    TraceScope trace_("bwd_convert_kernel", stream);
    bwd_convert_kernel<<<static_cast<unsigned>((nkv / 8 + 255) / 256), 256, 0, stream>>>(
        ws.dv_acc, static_cast<__nv_bfloat16*>(dv), nkv / 8, 1.0f);
  }
  return check_launch("bwd_convert_kernel");
}

}  // namespace msa
