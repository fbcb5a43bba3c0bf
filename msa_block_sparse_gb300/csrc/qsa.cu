// Narrow-block sparse attention ("[1/4] Add MiniMax-M3 support - #4581", Kernel
// tuning: the QSA layers of qwen3.8-next, 12 query heads per KV head, head dim
// 256, 4-token key blocks; "What": the tile map over blocks narrower or wider
// than a tile).  The semantics are those of the 128-token kernels with block 4:
// query token t (position p in its sequence) of KV group g attends to the keys
// j <= p of the blocks listed in sel[t, g, :].
//
// Data structures built per call:
//   masks  [T, Hkv, W] u32   bit b of row (t, g): block b is in sel[t, g]
//   plan   10-token query tiles (s, qt), heaviest first
//   ulist  per (query tile, g): count, then the 64-key tiles (16 blocks each)
//          holding a block selected by any of the tile's tokens ("tile map")
//
// Forward, persistent CTAs claiming the query tiles (heaviest first) from a
// counter.  Tile = 128 rows = 10 tokens x the 12 query heads of one KV head
// (rows 120..127 are padding):
//   warp 0 : TMA Q (4 x 64-column chunks) and K tiles (2-stage ring)
//   warp 2 : TMA V tiles (own 2-stage ring)
//   warp 1 : MMA  S_n = Q K_n^T (M 128, N 64, K 256) into one of two TMEM
//            buffers; O += P_n V_n (M 128, N 256, K 64), P_n read from TMEM
//   warps 4..7 : softmax, thread = row = TMEM lane: P = 2^(s scale log2e - m)
//            on the row's selected, causal keys (0 elsewhere), running max
//            rescaled only when it grows by more than 2^8; epilogue o = O / l.
#include "kernels.cuh"

namespace msa {

namespace {

constexpr int kQD = 256;                    // head dim
constexpr int kQG = 12;                     // query heads per KV head
constexpr int kQBlk = 4;                    // tokens per key block
constexpr int kQTok = 10;                   // tokens per query tile
constexpr int kQRows = kQTok * kQG;         // 120 live rows of the 128-row tile
constexpr int kQKeys = 64;                  // keys per key tile
constexpr int kQChunk = 128 * 128;          // 64-column chunk of a 128-row tile (bytes)
constexpr int kQTileBytes = 4 * kQChunk;    // 128 rows x 256 bf16
constexpr int kKChunk = kQKeys * 128;       // 64-column chunk of a 64-key tile
constexpr int kKTileBytes = 4 * kKChunk;    // 64 keys x 256 bf16
constexpr uint32_t kQIdS = idesc_bf16(128, 64, false, false);    // S = Q K^T
constexpr uint32_t kQIdPV = idesc_bf16(128, 256, false, true);   // O += P V
constexpr uint32_t kQColS = 256;            // O at columns 0..255, S buffers at 256, 320
constexpr float kQLog2e = 1.4426950408889634f;
constexpr float kQRescale = 8.0f;
constexpr int kQFwdThreads = 256;           // warps 0 Q/K, 1 MMA, 2 V, 3 idle, 4..7 softmax

// Work units (query tiles, or key-tile items) are claimed from a counter by
// one thread (the first producer) and passed to the other roles through a
// ring of slots: the second producer, the MMA thread and lane 0 of each of
// the four softmax / compute warps read every slot once.  -1 ends the loops.
constexpr int kRing = 4;
constexpr int kRingReaders = 6;
constexpr int kRingTimeout = -2;
struct ClaimRing {
  uint64_t full[kRing], empty[kRing];
  int id[kRing];
};
__device__ __forceinline__ void ring_init(ClaimRing& r) {
  for (int i = 0; i < kRing; ++i) {
    mbar_init(&r.full[i], 1);
    mbar_init(&r.empty[i], kRingReaders);
  }
}
// Publishes the id of the claimer's k-th unit; false if the wait ran out.
__device__ __forceinline__ bool ring_put(ClaimRing& r, uint32_t k, int id, uint32_t* status,
                                         uint32_t site) {
  const int sl = k % kRing;
  if (!mbar_wait(&r.empty[sl], ((k / kRing) & 1) ^ 1, status, site)) return false;
  r.id[sl] = id;
  mbar_arrive(&r.full[sl]);
  return true;
}
// The id of a reader's k-th unit (-1: none left; kRingTimeout: the wait ran out).
__device__ __forceinline__ int ring_get(ClaimRing& r, uint32_t k, uint32_t* status, uint32_t site) {
  const int sl = k % kRing;
  if (!mbar_wait(&r.full[sl], (k / kRing) & 1, status, site)) return kRingTimeout;
  const int id = r.id[sl];
  mbar_arrive(&r.empty[sl]);
  return id;
}

struct QsaFwdSmem {
  uint8_t q[kQTileBytes];
  uint8_t k[2][kKTileBytes];
  uint8_t v[2][kKTileBytes];
  uint64_t q_full, q_empty, k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2], o_free;
  ClaimRing ring;
  uint32_t tmem_base;
};
static_assert(sizeof(QsaFwdSmem) + 1024 <= 232448, "QSA forward shared memory");

__device__ __forceinline__ float qex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void umma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct QTile {
  int seq0, len, p0, ntok;
};

__device__ __forceinline__ QTile qsa_tile(const int2* tiles, const int32_t* cu, int ti) {
  const int2 pt = tiles[ti];
  QTile t;
  t.seq0 = cu[pt.x];
  t.len = cu[pt.x + 1] - t.seq0;
  t.p0 = pt.y * kQTok;
  t.ntok = min(kQTok, t.len - t.p0);
  return t;
}

// 16 selection bits of row `mrow` for key tile kt (blocks 16 kt .. 16 kt + 15)
__device__ __forceinline__ uint32_t tile_bits(const uint32_t* mrow, int kt) {
  return (__ldg(mrow + (kt >> 1)) >> ((kt & 1) * 16)) & 0xFFFFu;
}

}  // namespace

// One warp per (token, KV head) row, grid-striding: the bitmap of the row's
// selected blocks.  An id beyond the token's own block sets the bounds bit and is
// dropped; -1 entries are padding.  With vec (topk a multiple of 4, sel 16-byte
// aligned) every lane reads its ids as 16-byte vectors, all of the row's loads
// in flight at once.
__global__ void __launch_bounds__(256) qsa_mask_kernel(const int32_t* __restrict__ sel,
                                                       const int32_t* __restrict__ cu, int S,
                                                       int T, int Hkv, int topk, int W,
                                                       uint32_t* __restrict__ masks, int vec,
                                                       uint32_t* status) {
  pdl_enter();
  __shared__ uint32_t rows[8][kQsaMaxWords];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* row = rows[warp];
  const int nrows = T * Hkv;
  for (int rr = blockIdx.x * 8 + warp; rr < nrows; rr += gridDim.x * 8) {
    const int t = rr / Hkv;
    int lo = 0, hi = S;                        // sequence of t: cu[lo] <= t < cu[lo + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(cu + mid) <= t) lo = mid;
      else hi = mid;
    }
    const int own = (t - __ldg(cu + lo)) / kQBlk;
    for (int w = lane; w < W; w += 32) row[w] = 0u;
    __syncwarp();
    const int32_t* src = sel + static_cast<size_t>(rr) * topk;
    auto mark = [&](int b) {
      if (b < 0) return;
      if (b > own || b >= W * 32) {
        atomicOr(status, kStatusBounds);
        return;
      }
      atomicOr(&row[b >> 5], 1u << (b & 31));
    };
    if (vec) {
      constexpr int kV = kQsaMaxTopk / 128;     // 16-byte vectors per lane at most
      const int4* src4 = reinterpret_cast<const int4*>(src);
      int4 ids[kV];
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        const int j4 = lane + 32 * i;
        ids[i] = (4 * j4 < topk) ? __ldg(src4 + j4) : make_int4(-1, -1, -1, -1);
      }
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        mark(ids[i].x);
        mark(ids[i].y);
        mark(ids[i].z);
        mark(ids[i].w);
      }
    } else {
      for (int j = lane; j < topk; j += 32) mark(__ldg(src + j));
    }
    __syncwarp();
    uint32_t* dst = masks + static_cast<size_t>(rr) * W;
    for (int w = lane; w < W; w += 32) dst[w] = row[w];
    __syncwarp();
  }
}

// One warp per (query tile, KV head), grid-striding: the ascending list of key
// tiles that hold a block selected by any token of the tile.
__global__ void __launch_bounds__(256) qsa_union_kernel(const uint32_t* __restrict__ masks,
                                                        int W, const int32_t* __restrict__ cu,
                                                        const int2* __restrict__ tiles,
                                                        const int* __restrict__ num_tiles,
                                                        int Hkv, int ustride,
                                                        int* __restrict__ ulist,
                                                        int* __restrict__ tile_ctr,
                                                        uint32_t* status) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (blockIdx.x == 0)   // the persistent kernels claim query tiles from 0
    for (int i = threadIdx.x; i < Hkv; i += blockDim.x) tile_ctr[i] = 0;
  const int total = *num_tiles * Hkv;
  for (int gw = blockIdx.x * 8 + warp; gw < total; gw += gridDim.x * 8) {
    const int ti = gw / Hkv, g = gw % Hkv;
    const QTile t = qsa_tile(tiles, cu, ti);
    int* out = ulist + static_cast<size_t>(gw) * ustride;
    int nkt = t.ntok > 0 ? (t.p0 + t.ntok - 1) / kQKeys + 1 : 0;
    if (nkt > ustride - 1) {                  // a sequence longer than max_seqlen
      if (lane == 0) atomicOr(status, kStatusBounds);
      nkt = ustride - 1;
    }
    int base = 0;
    for (int c0 = 0; c0 < nkt; c0 += 32) {
      const int kt = c0 + lane;
      uint32_t bits = 0;
      if (kt < nkt)
        for (int j = 0; j < t.ntok; ++j)
          bits |= tile_bits(masks + (static_cast<size_t>(t.seq0 + t.p0 + j) * Hkv + g) * W, kt);
      const unsigned bal = __ballot_sync(0xffffffffu, bits != 0);
      if (bits) out[1 + base + __popc(bal & ((1u << lane) - 1u))] = kt;
      base += __popc(bal);
    }
    if (lane == 0) out[0] = base;
  }
}

__global__ void __launch_bounds__(kQFwdThreads, 1)
    qsa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const uint32_t* __restrict__ masks,
                   int W, const int* __restrict__ ulist, int ustride,
                   const int32_t* __restrict__ cu, const int2* __restrict__ tiles,
                   const int* __restrict__ num_tiles, int Hq, int Hkv, float scale,
                   __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int* __restrict__ ctr,
                      uint32_t* status) {
  pdl_enter();
  const int ntiles = *num_tiles;
  if (static_cast<int>(blockIdx.x) >= ntiles) return;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  QsaFwdSmem& sm = *reinterpret_cast<QsaFwdSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int g = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    mbar_init(&sm.o_free, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 1);
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], 128);
      mbar_init(&sm.pv_done[i], 1);
    }
    ring_init(sm.ring);
    fence_mbar_init();
  }
  if (warp >= 4) {
    // rows 120..127 of every Q chunk stay zero (the tensor copies fill 120 rows)
    const int i = tid - 128;                               // 0..127: 4 chunks x 1 KB
    uint4* pad = reinterpret_cast<uint4*>(sm.q + (i >> 5) * kQChunk + kQRows * 128);
    pad[(i & 31) * 2] = make_uint4(0u, 0u, 0u, 0u);
    pad[(i & 31) * 2 + 1] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
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
    // ------------------------------------------------------------ Q and K
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      uint32_t tc = 0, kc = 0;
      bool ok = true;
      int pending = atomicAdd(ctr + g, 1);
      for (uint32_t wu = 0; ok; ++wu) {
        const int ti = pending < ntiles ? pending : -1;
        if (!(ok = ring_put(sm.ring, wu, ti, status, 60))) break;
        if (ti < 0) break;
        pending = atomicAdd(ctr + g, 1);
        const QTile t = qsa_tile(tiles, cu, ti);
        const int* ul = ulist + (static_cast<size_t>(ti) * Hkv + g) * ustride;
        const int nk = __ldg(ul);
        if (nk == 0) continue;
        if (!(ok = mbar_wait(&sm.q_empty, (tc & 1) ^ 1, status, 1))) break;
        mbar_arrive_expect_tx(&sm.q_full, 4 * kQRows * 128);
        for (int c = 0; c < 4; ++c)
          tma_load_3d(sm.q + c * kQChunk, &tm_q, &sm.q_full, 64 * c, g * kQG, t.seq0 + t.p0);
        for (int i = 0; i < nk; ++i) {
          const int st = kc & 1;
          if (!(ok = mbar_wait(&sm.k_empty[st], ((kc >> 1) & 1) ^ 1, status, 2))) break;
          const int row = t.seq0 + __ldg(ul + 1 + i) * kQKeys;
          mbar_arrive_expect_tx(&sm.k_full[st], kKTileBytes);
          for (int c = 0; c < 4; ++c)
            tma_load_3d(sm.k[st] + c * kKChunk, &tm_k, &sm.k_full[st], 64 * c, g, row);
          ++kc;
        }
        ++tc;
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ V
    if (lane == 0) {
      prefetch_tmap(&tm_v);
      uint32_t vc = 0;
      bool ok = true;
      for (uint32_t wu = 0; ok; ++wu) {
        const int ti = ring_get(sm.ring, wu, status, 61);
        if (ti == kRingTimeout) ok = false;
        if (ti < 0) break;
        const QTile t = qsa_tile(tiles, cu, ti);
        const int* ul = ulist + (static_cast<size_t>(ti) * Hkv + g) * ustride;
        const int nk = __ldg(ul);
        for (int i = 0; i < nk; ++i) {
          const int st = vc & 1;
          if (!(ok = mbar_wait(&sm.v_empty[st], ((vc >> 1) & 1) ^ 1, status, 3))) break;
          const int row = t.seq0 + __ldg(ul + 1 + i) * kQKeys;
          mbar_arrive_expect_tx(&sm.v_full[st], kKTileBytes);
          for (int c = 0; c < 4; ++c)
            tma_load_3d(sm.v[st] + c * kKChunk, &tm_v, &sm.v_full[st], 64 * c, g, row);
          ++vc;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (elect_one()) {
      uint32_t tc = 0, kc = 0, vc = 0, n = 0;
      bool ok = true;
      const uint32_t qa = smem_u32(sm.q);
      for (uint32_t wu = 0; ok; ++wu) {
        const int ti = ring_get(sm.ring, wu, status, 61);
        if (ti == kRingTimeout) ok = false;
        if (ti < 0) break;
        const int nk = __ldg(ulist + (static_cast<size_t>(ti) * Hkv + g) * ustride);
        if (nk == 0) continue;
        if (!(ok = mbar_wait(&sm.q_full, tc & 1, status, 4))) break;
        tc_fence_after();
        const uint32_t n0 = n;
        for (int i = 0; ok && i <= nk; ++i) {
          if (i < nk) {
            const int st = kc & 1;
            if (!(ok = mbar_wait(&sm.k_full[st], (kc >> 1) & 1, status, 5))) break;
            // S buffer n & 1 last held P of step n - 2: its PV must be done
            if (n >= 2 && !(ok = mbar_wait(&sm.pv_done[n & 1], ((n - 2) >> 1) & 1, status, 6)))
              break;
            tc_fence_after();
            const uint32_t ka = smem_u32(sm.k[st]);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
              const uint32_t cq = (kk >> 2) * kQChunk + (kk & 3) * 32;
              const uint32_t ck = (kk >> 2) * kKChunk + (kk & 3) * 32;
              umma_bf16(tmem + kQColS + (n & 1) * 64, sdesc_sw128(qa + cq, 16, 1024),
                        sdesc_sw128(ka + ck, 16, 1024), kQIdS, kk > 0);
            }
            umma_commit(&sm.s_full[n & 1]);
            umma_commit(&sm.k_empty[st]);
            if (i == nk - 1) umma_commit(&sm.q_empty);   // Q is free once these are done
            ++kc;
            ++n;
          }
          if (i > 0) {
            const uint32_t j = n0 + i - 1;
            const int st = vc & 1;
            if (!(ok = mbar_wait(&sm.p_full[j & 1], (j >> 1) & 1, status, 7))) break;
            if (!(ok = mbar_wait(&sm.v_full[st], (vc >> 1) & 1, status, 8))) break;
            // the first PV of a tile overwrites O: the previous epilogue must be done
            if (i == 1 && tc > 0 && !(ok = mbar_wait(&sm.o_free, (tc - 1) & 1, status, 9)))
              break;
            tc_fence_after();
            const uint32_t va = smem_u32(sm.v[st]);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_tmem_a(tmem, tmem + kQColS + (j & 1) * 64 + kk * 8,
                          sdesc_sw128(va + kk * 2048, kKChunk, 1024), kQIdPV,
                          (i > 1 || kk > 0) ? 1u : 0u);
            umma_commit(&sm.pv_done[j & 1]);
            umma_commit(&sm.v_empty[st]);
            ++vc;
          }
        }
        ++tc;
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int tok = r / kQG, hd = r - (r / kQG) * kQG;
    const uint32_t trow = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = scale * kQLog2e;
    uint32_t tc = 0, n = 0;
    bool ok = true;
    for (uint32_t wu = 0; ok; ++wu) {
      int ti = 0;
      if (lane == 0) ti = ring_get(sm.ring, wu, status, 62);
      ti = __shfl_sync(0xffffffffu, ti, 0);
      if (ti == kRingTimeout) ok = false;
      if (ti < 0) break;
      const QTile t = qsa_tile(tiles, cu, ti);
      const int* ul = ulist + (static_cast<size_t>(ti) * Hkv + g) * ustride;
      const int nk = __ldg(ul);
      const bool valid = r < kQRows && tok < t.ntok;
      const int pos = t.p0 + tok;
      const size_t orow = (static_cast<size_t>(t.seq0 + pos) * Hq + g * kQG + hd);
      if (nk == 0) {
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(o + orow * kQD);
          for (int c = 0; c < kQD / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
          lse[orow] = -INFINITY;
        }
        continue;
      }
      const uint32_t* mrow = masks + (static_cast<size_t>(t.seq0 + (valid ? pos : 0)) * Hkv + g) * W;
      float m = -INFINITY, l = 0.f;
      for (int i = 0; i < nk; ++i) {
        const int kt = __ldg(ul + 1 + i);
        const uint32_t bits = valid ? tile_bits(mrow, kt) : 0u;
        const int kmax = pos - kt * kQKeys;          // last causal column of this key tile
        const uint32_t sbuf = tmem + kQColS + (n & 1) * 64 + trow;
        if (!(ok = mbar_wait(&sm.s_full[n & 1], (n >> 1) & 1, status, 10))) break;
        __syncwarp();
        tc_fence_after();
        uint32_t sv[64];
        tmem_ld32(sbuf, sv);
        tmem_ld32(sbuf + 32, sv + 32);
        tmem_ld_wait();
        bool resc = false, live = false;
        float mu = m, rs = 0.f;
        uint32_t pk[32];
        if (bits != 0u && kmax >= 0) {
          float x[64];
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const bool keep = ((bits >> (j >> 2)) & 1u) && j <= kmax;
            x[j] = keep ? __uint_as_float(sv[j]) : -INFINITY;
          }
          float mx8[8];
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8) {
            const float* xi = x + 8 * q8;
            mx8[q8] = fmaxf(max3f(max3f(max3f(xi[0], xi[1], xi[2]), xi[3], xi[4]), xi[5], xi[6]),
                            xi[7]);
          }
          const float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]),
                                 fmaxf(mx8[6], mx8[7]));
          live = mx != -INFINITY;
          if (live) {
            const float mnew = fmaxf(m, mx * sl2);
            resc = mnew > m + kQRescale;
            mu = resc ? mnew : m;
            const float2 sl2v = make_float2(sl2, sl2), nmu = make_float2(-mu, -mu);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int j2 = 0; j2 < 32; ++j2) {
              const float2 y = ffma2(make_float2(x[2 * j2], x[2 * j2 + 1]), sl2v, nmu);
              const float2 pe = make_float2(qex2(y.x), qex2(y.y));
              acc[j2 & 3] = fadd2(acc[j2 & 3], pe);
              pk[j2] = pack_bf16x2(pe.x, pe.y);
            }
            const float2 a01 = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
            rs = a01.x + a01.y;
          }
        }
        if (!live) {
#pragma unroll
          for (int j = 0; j < 32; ++j) pk[j] = 0u;
        }
        const bool need = resc && m != -INFINITY;
        if (__any_sync(0xffffffffu, need)) {
          // O is stable once the PV of the previous step is done
          if (!(ok = mbar_wait(&sm.pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, status, 11))) break;
          __syncwarp();
          tc_fence_after();
          const float alpha = need ? qex2(m - mu) : 1.f;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + trow + c * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
            tmem_st16(tmem + trow + c * 32, v);
            tmem_st16(tmem + trow + c * 32 + 16, v + 16);
          }
        }
        if (live) {
          l = (m == -INFINITY) ? rs : (resc ? l * qex2(m - mu) : l) + rs;
          m = mu;
        }
        tmem_st16(sbuf, pk);
        tmem_st16(sbuf + 16, pk + 16);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full[n & 1]);
        ++n;
      }
      if (!ok) break;
      // ---- epilogue: the tile's last PV completes after all earlier ones
      if (!(ok = mbar_wait(&sm.pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, status, 12))) break;
      __syncwarp();
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(o + orow * kQD);
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t a[32];
        tmem_ld32(tmem + trow + c * 32, a);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 pk4;
            pk4.x = pack_bf16x2(__uint_as_float(a[8 * q4 + 0]) * inv, __uint_as_float(a[8 * q4 + 1]) * inv);
            pk4.y = pack_bf16x2(__uint_as_float(a[8 * q4 + 2]) * inv, __uint_as_float(a[8 * q4 + 3]) * inv);
            pk4.z = pack_bf16x2(__uint_as_float(a[8 * q4 + 4]) * inv, __uint_as_float(a[8 * q4 + 5]) * inv);
            pk4.w = pack_bf16x2(__uint_as_float(a[8 * q4 + 6]) * inv, __uint_as_float(a[8 * q4 + 7]) * inv);
            dst[4 * c + q4] = pk4;
          }
        }
      }
      if (valid) lse[orow] = (l > 0.f) ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
      tc_fence_before();
      mbar_arrive(&sm.o_free);
      ++tc;
    }
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- backward
// Two passes that recompute S and dP (head dim 256 leaves too little tensor
// memory to keep dQ, dK and dV accumulators beside them):
//   dQ  pass, query-tile major (the forward's tiles and tile map): per key
//       tile S, dP into TMEM, dS = P (dP - Delta) back into S's columns as
//       bf16, dQ += dS K with dS read from TMEM; dQ stays in TMEM for the tile.
//   dKV pass, key-tile major: item = (64-key tile, window of 128 query tiles);
//       per query tile S, dP into TMEM, P and dS written to shared memory,
//       dV^T += dO^T P and dK^T += Q^T dS (M = 128 head-dim rows, N = 64 keys),
//       so both accumulators fit beside S and dP.  A key tile's windows are
//       summed with fp32 reductions, then converted to bf16.

namespace {

constexpr int kQWin = 128;                  // query tiles per dKV item
constexpr int kQBwdThreads = 256;
constexpr uint32_t kQIdDq = idesc_bf16(128, 256, false, true);   // dQ += dS K
constexpr uint32_t kQIdKV = idesc_bf16(128, 64, true, true);     // dV^T += dO^T P, dK^T += Q^T dS

struct QsaDqSmem {
  uint8_t q[kQTileBytes];
  uint8_t dout[kQTileBytes];
  uint8_t k[2][kKTileBytes];
  uint8_t v[kKTileBytes];
  uint64_t qd_full, qd_empty, k_full[2], k_empty[2], v_full, v_empty;
  uint64_t s_full[2], ds_full[2], dq_done[2], dq_free;
  ClaimRing ring;
  uint32_t tmem_base;
};
static_assert(sizeof(QsaDqSmem) + 1024 <= 232448, "QSA dQ shared memory");

struct QsaDkvSmem {
  uint8_t q[kQTileBytes];
  uint8_t dout[kQTileBytes];
  uint8_t k[kKTileBytes];
  uint8_t v[kKTileBytes];
  uint8_t p[128 * 128];                     // P, rows x 64 keys, 128B-swizzled
  uint8_t ds[128 * 128];                    // dS, same layout
  // Q and dO move as two halves of 128 head-dim columns each: half h is what
  // the h-th dK^T / dV^T MMA reads, so the next tile's half h loads as soon as
  // that MMA is done
  uint64_t kv_full, kv_empty, q_full[2], q_empty[2], do_full[2], do_empty[2];
  uint64_t s_full, pds_full, pds_empty, acc_full, acc_free;
  ClaimRing ring;
  uint32_t tmem_base;
};
static_assert(sizeof(QsaDkvSmem) + 1024 <= 232448, "QSA dK/dV shared memory");

// Zero rows 120..127 of the four chunks of a 128-row tile (128 threads).
__device__ __forceinline__ void zero_pad_rows(uint8_t* tile, int i) {
  uint4* pad = reinterpret_cast<uint4*>(tile + (i >> 5) * kQChunk + kQRows * 128);
  pad[(i & 31) * 2] = make_uint4(0u, 0u, 0u, 0u);
  pad[(i & 31) * 2 + 1] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

// lsd[t Hq + h] = (-lse log2 e, -Delta), Delta = sum_d dout o; 16 lanes per row.
__global__ void __launch_bounds__(256) qsa_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        const float* __restrict__ lse,
                                                        float2* __restrict__ lsd, size_t rows) {
  pdl_enter();
  const int sub = threadIdx.x & 15;
  // warp-uniform loop: each warp takes two rows per pass, so every lane of the
  // warp reaches the shuffles
  const size_t warp0 = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const size_t nwarps = (static_cast<size_t>(gridDim.x) * blockDim.x) >> 5;
  for (size_t base = 2 * warp0; base < rows; base += 2 * nwarps) {
    const size_t row = base + ((threadIdx.x >> 4) & 1);
    const bool live = row < rows;
    uint4 a0 = make_uint4(0u, 0u, 0u, 0u), a1 = a0, b0 = a0, b1 = a0;
    if (live) {
      const uint4* a = reinterpret_cast<const uint4*>(o + row * kQD) + sub * 2;
      const uint4* b = reinterpret_cast<const uint4*>(dout + row * kQD) + sub * 2;
      a0 = __ldcs(a);
      a1 = __ldcs(a + 1);
      b0 = __ldcs(b);
      b1 = __ldcs(b + 1);
    }
    float acc = 0.f;
    const __nv_bfloat162* x0 = reinterpret_cast<const __nv_bfloat162*>(&a0);
    const __nv_bfloat162* x1 = reinterpret_cast<const __nv_bfloat162*>(&a1);
    const __nv_bfloat162* y0 = reinterpret_cast<const __nv_bfloat162*>(&b0);
    const __nv_bfloat162* y1 = reinterpret_cast<const __nv_bfloat162*>(&b1);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 p0 = __bfloat1622float2(x0[j]), q0 = __bfloat1622float2(y0[j]);
      const float2 p1 = __bfloat1622float2(x1[j]), q1 = __bfloat1622float2(y1[j]);
      acc = fmaf(p0.x, q0.x, fmaf(p0.y, q0.y, fmaf(p1.x, q1.x, fmaf(p1.y, q1.y, acc))));
    }
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (sub == 0 && live) lsd[row] = make_float2(-__ldg(lse + row) * kQLog2e, -acc);
  }
}

// One CTA: the dKV work items (s, key tile kt, window w) of every sequence, in
// sequence order; windows that start before the key tile's first query tile
// are listed too and end up empty.
__global__ void __launch_bounds__(1024) qsa_items_kernel(const int32_t* __restrict__ cu, int S,
                                                         int4* __restrict__ items,
                                                         int* __restrict__ num_items,
                                                         int max_items, uint32_t* status) {
  pdl_enter();
  int base = 0;
  for (int s = 0; s < S; ++s) {
    const int len = __ldg(cu + s + 1) - __ldg(cu + s);
    if (len <= 0) continue;
    const int nkt = (len + kQKeys - 1) / kQKeys;
    const int nw = ((len + kQTok - 1) / kQTok + kQWin - 1) / kQWin;
    const int n = nkt * nw;
    for (int j = threadIdx.x; j < n; j += blockDim.x)
      if (base + j < max_items) items[base + j] = make_int4(s, j / nw, j % nw, 0);
    base += n;
  }
  if (threadIdx.x == 0) {
    *num_items = base < max_items ? base : max_items;
    if (base > max_items) atomicOr(status, kStatusBounds);
  }
}

// One warp per (item, KV head), grid-striding: the query tiles of the item's
// window that select a block of its key tile, ascending.
__global__ void __launch_bounds__(256) qsa_kvlist_kernel(const uint32_t* __restrict__ masks,
                                                         int W, const int32_t* __restrict__ cu,
                                                         const int4* __restrict__ items,
                                                         const int* __restrict__ num_items,
                                                         int Hkv, int* __restrict__ klist) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = *num_items * Hkv;
  for (int gw = blockIdx.x * 8 + warp; gw < total; gw += gridDim.x * 8) {
    const int4 it = items[gw / Hkv];
    const int g = gw % Hkv;
    const int seq0 = __ldg(cu + it.x), len = __ldg(cu + it.x + 1) - seq0;
    const int nqt = (len + kQTok - 1) / kQTok;
    const int lo = max(it.z * kQWin, (it.y * kQKeys) / kQTok);
    const int hi = min(it.z * kQWin + kQWin, nqt);
    int* out = klist + static_cast<size_t>(gw) * (1 + kQWin);
    int base = 0;
    for (int c0 = lo; c0 < hi; c0 += 32) {
      const int qt = c0 + lane;
      uint32_t bits = 0;
      if (qt < hi) {
        const int p1 = min(qt * kQTok + kQTok, len);
        for (int p = qt * kQTok; p < p1; ++p)
          bits |= tile_bits(masks + (static_cast<size_t>(seq0 + p) * Hkv + g) * W, it.y);
      }
      const unsigned bal = __ballot_sync(0xffffffffu, bits != 0);
      if (bits) out[1 + base + __popc(bal & ((1u << lane) - 1u))] = qt;
      base += __popc(bal);
    }
    if (lane == 0) out[0] = base;
  }
}

// One CTA per KV head: the non-empty items ordered by their number of query
// tiles, largest first (counting sort), so that CTAs striding over the order
// get nearly equal work.
__global__ void __launch_bounds__(1024) qsa_order_kernel(const int* __restrict__ klist,
                                                         const int* __restrict__ num_items,
                                                         int Hkv, int max_items,
                                                         int* __restrict__ order,
                                                         int* __restrict__ num_busy,
                                                         int* __restrict__ item_ctr) {
  pdl_enter();
  if (threadIdx.x == 0) item_ctr[blockIdx.x] = 0;   // the dK/dV kernel claims items from 0
  __shared__ int hist[kQWin + 1];
  __shared__ int start[kQWin + 1];
  const int g = blockIdx.x;
  const int n = *num_items;
  for (int c = threadIdx.x; c <= kQWin; c += blockDim.x) hist[c] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    atomicAdd(&hist[min(klist[(static_cast<size_t>(i) * Hkv + g) * (1 + kQWin)], kQWin)], 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int c = kQWin; c >= 1; --c) {
      start[c] = acc;
      acc += hist[c];
    }
    num_busy[g] = acc;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int c = min(klist[(static_cast<size_t>(i) * Hkv + g) * (1 + kQWin)], kQWin);
    if (c > 0) order[static_cast<size_t>(g) * max_items + atomicAdd(&start[c], 1)] = i;
  }
}

__global__ void __launch_bounds__(kQBwdThreads, 1)
    qsa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const uint32_t* __restrict__ masks, int W, const int* __restrict__ ulist,
                      int ustride, const float2* __restrict__ lsd, const int32_t* __restrict__ cu,
                      const int2* __restrict__ tiles, const int* __restrict__ num_tiles, int Hq,
                      int Hkv, float scale, __nv_bfloat16* __restrict__ dq, int* __restrict__ ctr,
                      uint32_t* status) {
  pdl_enter();
  const int ntiles = *num_tiles;
  if (static_cast<int>(blockIdx.x) >= ntiles) return;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  QsaDqSmem& sm = *reinterpret_cast<QsaDqSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int g = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr uint32_t kColDq = 0, kColS = 256, kColDp = 384;

  if (tid == 0) {
    mbar_init(&sm.qd_full, 1);
    mbar_init(&sm.qd_empty, 1);
    mbar_init(&sm.v_full, 1);
    mbar_init(&sm.v_empty, 1);
    mbar_init(&sm.dq_free, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.ds_full[i], 128);
      mbar_init(&sm.dq_done[i], 1);
    }
    ring_init(sm.ring);
    fence_mbar_init();
  }
  if (warp >= 4) {
    zero_pad_rows(sm.q, tid - 128);
    zero_pad_rows(sm.dout, tid - 128);
    fence_proxy_async_smem();
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
    // ------------------------------------------------------------ Q, dO and K
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_do);
      prefetch_tmap(&tm_k);
      uint32_t tc = 0, kc = 0;
      bool ok = true;
      int pending = atomicAdd(ctr + g, 1);
      for (uint32_t wu = 0; ok; ++wu) {
        const int ti = pending < ntiles ? pending : -1;
        if (!(ok = ring_put(sm.ring, wu, ti, status, 60))) break;
        if (ti < 0) break;
        pending = atomicAdd(ctr + g, 1);
        const QTile t = qsa_tile(tiles, cu, ti);
        const int* ul = ulist + (static_cast<size_t>(ti) * Hkv + g) * ustride;
        const int nk = __ldg(ul);
        if (nk == 0) continue;
        if (!(ok = mbar_wait(&sm.qd_empty, (tc & 1) ^ 1, status, 21))) break;
        mbar_arrive_expect_tx(&sm.qd_full, 8 * kQRows * 128);
        for (int c = 0; c < 4; ++c) {
          tma_load_3d(sm.q + c * kQChunk, &tm_q, &sm.qd_full, 64 * c, g * kQG, t.seq0 + t.p0);
          tma_load_3d(sm.dout + c * kQChunk, &tm_do, &sm.qd_full, 64 * c, g * kQG,
                      t.seq0 + t.p0);
        }
        for (int i = 0; i < nk; ++i) {
          const int st = kc & 1;
          if (!(ok = mbar_wait(&sm.k_empty[st], ((kc >> 1) & 1) ^ 1, status, 22))) break;
          const int row = t.seq0 + __ldg(ul + 1 + i) * kQKeys;
          mbar_arrive_expect_tx(&sm.k_full[st], kKTileBytes);
          for (int c = 0; c < 4; ++c)
            tma_load_3d(sm.k[st] + c * kKChunk, &tm_k, &sm.k_full[st], 64 * c, g, row);
          ++kc;
        }
        ++tc;
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ V (one stage)
    if (lane == 0) {
      prefetch_tmap(&tm_v);
      uint32_t vc = 0;
      bool ok = true;
      for (uint32_t wu = 0; ok; ++wu) {
        const int ti = ring_get(sm.ring, wu, status, 61);
        if (ti == kRingTimeout) ok = false;
        if (ti < 0) break;
        const QTile t = qsa_tile(tiles, cu, ti);
        const int* ul = ulist + (static_cast<size_t>(ti) * Hkv + g) * ustride;
        const int nk = __ldg(ul);
        for (int i = 0; i < nk; ++i) {
          if (!(ok = mbar_wait(&sm.v_empty, (vc & 1) ^ 1, status, 23))) break;
          const int row = t.seq0 + __ldg(ul + 1 + i) * kQKeys;
          mbar_arrive_expect_tx(&sm.v_full, kKTileBytes);
          for (int c = 0; c < 4; ++c)
            tma_load_3d(sm.v + c * kKChunk, &tm_v, &sm.v_full, 64 * c, g, row);
          ++vc;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (elect_one()) {
      uint32_t tc = 0, kc = 0, kq = 0, vc = 0, n = 0;
      bool ok = true;
      const uint32_t qa = smem_u32(sm.q), da = smem_u32(sm.dout), va = smem_u32(sm.v);
      for (uint32_t wu = 0; ok; ++wu) {
        const int ti = ring_get(sm.ring, wu, status, 61);
        if (ti == kRingTimeout) ok = false;
        if (ti < 0) break;
        const int nk = __ldg(ulist + (static_cast<size_t>(ti) * Hkv + g) * ustride);
        if (nk == 0) continue;
        if (!(ok = mbar_wait(&sm.qd_full, tc & 1, status, 24))) break;
        tc_fence_after();
        const uint32_t n0 = n;
        for (int i = 0; ok && i <= nk; ++i) {
          if (i < nk) {
            const int st = kc & 1;
            // S / dP buffers n & 1 last held step n - 2: its dQ MMA must be done
            if (n >= 2 && !(ok = mbar_wait(&sm.dq_done[n & 1], ((n - 2) >> 1) & 1, status, 27)))
              break;
            // dP first: the single V stage is released as early as possible
            if (!(ok = mbar_wait(&sm.v_full, vc & 1, status, 26))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
              const uint32_t cq = (kk >> 2) * kQChunk + (kk & 3) * 32;
              const uint32_t ck = (kk >> 2) * kKChunk + (kk & 3) * 32;
              umma_bf16(tmem + kColDp + (n & 1) * 64, sdesc_sw128(da + cq, 16, 1024),
                        sdesc_sw128(va + ck, 16, 1024), kQIdS, kk > 0);
            }
            umma_commit(&sm.v_empty);
            if (!(ok = mbar_wait(&sm.k_full[st], (kc >> 1) & 1, status, 25))) break;
            tc_fence_after();
            const uint32_t ka = smem_u32(sm.k[st]);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
              const uint32_t cq = (kk >> 2) * kQChunk + (kk & 3) * 32;
              const uint32_t ck = (kk >> 2) * kKChunk + (kk & 3) * 32;
              umma_bf16(tmem + kColS + (n & 1) * 64, sdesc_sw128(qa + cq, 16, 1024),
                        sdesc_sw128(ka + ck, 16, 1024), kQIdS, kk > 0);
            }
            umma_commit(&sm.s_full[n & 1]);
            if (i == nk - 1) umma_commit(&sm.qd_empty);
            ++kc;
            ++vc;
            ++n;
          }
          if (i > 0) {
            const uint32_t j = n0 + i - 1;
            const int st = kq & 1;
            if (!(ok = mbar_wait(&sm.ds_full[j & 1], (j >> 1) & 1, status, 28))) break;
            if (i == 1 && tc > 0 && !(ok = mbar_wait(&sm.dq_free, (tc - 1) & 1, status, 29)))
              break;
            tc_fence_after();
            const uint32_t ka = smem_u32(sm.k[st]);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_tmem_a(tmem + kColDq, tmem + kColS + (j & 1) * 64 + kk * 8,
                          sdesc_sw128(ka + kk * 2048, kKChunk, 1024), kQIdDq,
                          (i > 1 || kk > 0) ? 1u : 0u);
            umma_commit(&sm.dq_done[j & 1]);
            umma_commit(&sm.k_empty[st]);
            ++kq;
          }
        }
        ++tc;
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ dS and epilogue
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int tok = r / kQG, hd = r - (r / kQG) * kQG;
    const uint32_t trow = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = scale * kQLog2e;
    uint32_t tc = 0, n = 0;
    bool ok = true;
    for (uint32_t wu = 0; ok; ++wu) {
      int ti = 0;
      if (lane == 0) ti = ring_get(sm.ring, wu, status, 62);
      ti = __shfl_sync(0xffffffffu, ti, 0);
      if (ti == kRingTimeout) ok = false;
      if (ti < 0) break;
      const QTile t = qsa_tile(tiles, cu, ti);
      const int* ul = ulist + (static_cast<size_t>(ti) * Hkv + g) * ustride;
      const int nk = __ldg(ul);
      const bool valid = r < kQRows && tok < t.ntok;
      const int pos = t.p0 + tok;
      const size_t qrow = static_cast<size_t>(t.seq0 + pos) * Hq + g * kQG + hd;
      if (nk == 0) {
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(dq + qrow * kQD);
          for (int c = 0; c < kQD / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      const uint32_t* mrow = masks + (static_cast<size_t>(t.seq0 + (valid ? pos : 0)) * Hkv + g) * W;
      const float2 ld = valid ? __ldg(lsd + qrow) : make_float2(0.f, 0.f);
      for (int i = 0; i < nk; ++i) {
        const int kt = __ldg(ul + 1 + i);
        const uint32_t bits = valid ? tile_bits(mrow, kt) : 0u;
        const int kmax = pos - kt * kQKeys;
        const uint32_t sbuf = tmem + kColS + (n & 1) * 64 + trow;
        const uint32_t pbuf = tmem + kColDp + (n & 1) * 64 + trow;
        if (!(ok = mbar_wait(&sm.s_full[n & 1], (n >> 1) & 1, status, 30))) break;
        __syncwarp();
        tc_fence_after();
        uint32_t sv[64], dv[64];
        tmem_ld32(sbuf, sv);
        tmem_ld32(sbuf + 32, sv + 32);
        tmem_ld32(pbuf, dv);
        tmem_ld32(pbuf + 32, dv + 32);
        tmem_ld_wait();
        uint32_t pk[32];
        // keys in pairs: one selection bit per pair, fp32 math two lanes at a time
        const float2 sl2v = make_float2(sl2, sl2), lxv = make_float2(ld.x, ld.x),
                     lyv = make_float2(ld.y, ld.y);
#pragma unroll
        for (int j2 = 0; j2 < 32; ++j2) {
          const int j = 2 * j2;
          const bool blk = (bits >> (j >> 2)) & 1u;
          const float2 y = ffma2(make_float2(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])),
                                 sl2v, lxv);
          const float2 pe = make_float2(qex2(y.x), qex2(y.y));
          float2 dd = fmul2(
              pe, fadd2(make_float2(__uint_as_float(dv[j]), __uint_as_float(dv[j + 1])), lyv));
          dd.x = (blk && j <= kmax) ? dd.x : 0.f;
          dd.y = (blk && j + 1 <= kmax) ? dd.y : 0.f;
          pk[j2] = pack_bf16x2(dd.x, dd.y);
        }
        tmem_st16(sbuf, pk);
        tmem_st16(sbuf + 16, pk + 16);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.ds_full[n & 1]);
        ++n;
      }
      if (!ok) break;
      if (!(ok = mbar_wait(&sm.dq_done[(n - 1) & 1], ((n - 1) >> 1) & 1, status, 31))) break;
      __syncwarp();
      tc_fence_after();
      uint4* dst = reinterpret_cast<uint4*>(dq + qrow * kQD);
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t a[32];
        tmem_ld32(tmem + kColDq + trow + c * 32, a);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 pk4;
            pk4.x = pack_bf16x2(__uint_as_float(a[8 * q4 + 0]) * scale, __uint_as_float(a[8 * q4 + 1]) * scale);
            pk4.y = pack_bf16x2(__uint_as_float(a[8 * q4 + 2]) * scale, __uint_as_float(a[8 * q4 + 3]) * scale);
            pk4.z = pack_bf16x2(__uint_as_float(a[8 * q4 + 4]) * scale, __uint_as_float(a[8 * q4 + 5]) * scale);
            pk4.w = pack_bf16x2(__uint_as_float(a[8 * q4 + 6]) * scale, __uint_as_float(a[8 * q4 + 7]) * scale);
            dst[4 * c + q4] = pk4;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.dq_free);
      ++tc;
    }
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

__global__ void __launch_bounds__(kQBwdThreads, 1)
    qsa_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const uint32_t* __restrict__ masks, int W, const int* __restrict__ klist,
                       const float2* __restrict__ lsd, const int32_t* __restrict__ cu,
                       const int4* __restrict__ items, const int* __restrict__ order,
                       const int* __restrict__ num_busy, int max_items, int Hq, int Hkv,
                       float scale, float* __restrict__ dk_acc, float* __restrict__ dv_acc,
                       int* __restrict__ ctr,
                      uint32_t* status) {
  pdl_enter();
  const int nitems = num_busy[blockIdx.y];
  if (static_cast<int>(blockIdx.x) >= nitems) return;
  const int* ord = order + static_cast<size_t>(blockIdx.y) * max_items;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  QsaDkvSmem& sm = *reinterpret_cast<QsaDkvSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int g = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr uint32_t kColS = 0, kColDp = 64, kColDv = 256, kColDk = 384;

  if (tid == 0) {
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    for (int hf = 0; hf < 2; ++hf) {
      mbar_init(&sm.q_full[hf], 1);
      mbar_init(&sm.q_empty[hf], 1);
      mbar_init(&sm.do_full[hf], 1);
      mbar_init(&sm.do_empty[hf], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.pds_full, 128);
    mbar_init(&sm.pds_empty, 1);
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_free, 128);
    ring_init(sm.ring);
    fence_mbar_init();
  }
  if (warp >= 4) {
    // the padding rows take part in the row-contracting MMAs: keep them zero
    zero_pad_rows(sm.q, tid - 128);
    zero_pad_rows(sm.dout, tid - 128);
    fence_proxy_async_smem();
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
    // ------------------------------------------------------------ K, V, Q
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      uint32_t ic = 0, qc = 0;
      bool ok = true;
      int pending = atomicAdd(ctr + g, 1);
      for (uint32_t wu = 0; ok; ++wu) {
        const int jt = pending < nitems ? pending : -1;
        if (!(ok = ring_put(sm.ring, wu, jt, status, 60))) break;
        if (jt < 0) break;
        pending = atomicAdd(ctr + g, 1);
        const int it = __ldg(ord + jt);
        const int* kl = klist + (static_cast<size_t>(it) * Hkv + g) * (1 + kQWin);
        const int nq = __ldg(kl);
        if (nq == 0) continue;
        const int4 item = items[it];
        const int seq0 = __ldg(cu + item.x);
        if (!(ok = mbar_wait(&sm.kv_empty, (ic & 1) ^ 1, status, 41))) break;
        mbar_arrive_expect_tx(&sm.kv_full, 2 * kKTileBytes);
        for (int c = 0; c < 4; ++c) {
          tma_load_3d(sm.k + c * kKChunk, &tm_k, &sm.kv_full, 64 * c, g, seq0 + item.y * kQKeys);
          tma_load_3d(sm.v + c * kKChunk, &tm_v, &sm.kv_full, 64 * c, g, seq0 + item.y * kQKeys);
        }
        for (int i = 0; ok && i < nq; ++i) {
          const int qt = __ldg(kl + 1 + i);
          for (int hf = 0; hf < 2; ++hf) {
            if (!(ok = mbar_wait(&sm.q_empty[hf], (qc & 1) ^ 1, status, 42))) break;
            mbar_arrive_expect_tx(&sm.q_full[hf], 2 * kQRows * 128);
            for (int c = 2 * hf; c < 2 * hf + 2; ++c)
              tma_load_3d(sm.q + c * kQChunk, &tm_q, &sm.q_full[hf], 64 * c, g * kQG,
                          seq0 + qt * kQTok);
          }
          ++qc;
        }
        ++ic;
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ dO
    if (lane == 0) {
      prefetch_tmap(&tm_do);
      uint32_t dc = 0;
      bool ok = true;
      for (uint32_t wu = 0; ok; ++wu) {
        const int jt = ring_get(sm.ring, wu, status, 61);
        if (jt == kRingTimeout) ok = false;
        if (jt < 0) break;
        const int it = __ldg(ord + jt);
        const int* kl = klist + (static_cast<size_t>(it) * Hkv + g) * (1 + kQWin);
        const int nq = __ldg(kl);
        if (nq == 0) continue;
        const int seq0 = __ldg(cu + items[it].x);
        for (int i = 0; ok && i < nq; ++i) {
          const int qt = __ldg(kl + 1 + i);
          for (int hf = 0; hf < 2; ++hf) {
            if (!(ok = mbar_wait(&sm.do_empty[hf], (dc & 1) ^ 1, status, 43))) break;
            mbar_arrive_expect_tx(&sm.do_full[hf], 2 * kQRows * 128);
            for (int c = 2 * hf; c < 2 * hf + 2; ++c)
              tma_load_3d(sm.dout + c * kQChunk, &tm_do, &sm.do_full[hf], 64 * c, g * kQG,
                          seq0 + qt * kQTok);
          }
          ++dc;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (elect_one()) {
      uint32_t ic = 0, n = 0;
      bool ok = true;
      const uint32_t qa = smem_u32(sm.q), da = smem_u32(sm.dout), ka = smem_u32(sm.k),
                     va = smem_u32(sm.v), pa = smem_u32(sm.p), sa = smem_u32(sm.ds);
      for (uint32_t wu = 0; ok; ++wu) {
        const int jt = ring_get(sm.ring, wu, status, 61);
        if (jt == kRingTimeout) ok = false;
        if (jt < 0) break;
        const int it = __ldg(ord + jt);
        const int nq = __ldg(klist + (static_cast<size_t>(it) * Hkv + g) * (1 + kQWin));
        if (nq == 0) continue;
        if (!(ok = mbar_wait(&sm.kv_full, ic & 1, status, 44))) break;
        for (int i = 0; ok && i < nq; ++i, ++n) {
          // S over the two Q halves as they land, then dP over the dO halves
          for (int hf = 0; ok && hf < 2; ++hf) {
            if (!(ok = mbar_wait(&sm.q_full[hf], n & 1, status, 45))) break;
            tc_fence_after();
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) {
              const int kk = 8 * hf + k8;
              const uint32_t cq = (kk >> 2) * kQChunk + (kk & 3) * 32;
              const uint32_t ck = (kk >> 2) * kKChunk + (kk & 3) * 32;
              umma_bf16(tmem + kColS, sdesc_sw128(qa + cq, 16, 1024),
                        sdesc_sw128(ka + ck, 16, 1024), kQIdS, kk > 0);
            }
          }
          for (int hf = 0; ok && hf < 2; ++hf) {
            if (!(ok = mbar_wait(&sm.do_full[hf], n & 1, status, 46))) break;
            tc_fence_after();
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) {
              const int kk = 8 * hf + k8;
              const uint32_t cq = (kk >> 2) * kQChunk + (kk & 3) * 32;
              const uint32_t ck = (kk >> 2) * kKChunk + (kk & 3) * 32;
              umma_bf16(tmem + kColDp, sdesc_sw128(da + cq, 16, 1024),
                        sdesc_sw128(va + ck, 16, 1024), kQIdS, kk > 0);
            }
          }
          if (!ok) break;
          umma_commit(&sm.s_full);
          if (i == nq - 1) umma_commit(&sm.kv_empty);    // K, V are free once S, dP are done
          if (!(ok = mbar_wait(&sm.pds_full, n & 1, status, 47))) break;
          // the item's first product overwrites the accumulators: the previous
          // item's epilogue must have read them
          if (i == 0 && ic > 0 && !(ok = mbar_wait(&sm.acc_free, (ic - 1) & 1, status, 48)))
            break;
          tc_fence_after();
          // dK first, one head-dim half at a time: each Q half is released as
          // soon as its MMAs are done, so the next tile's Q (which its S needs
          // before its dP needs dO) loads while the rest runs
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16(tmem + kColDk + hf * 64,
                        sdesc_sw128(qa + hf * 2 * kQChunk + kk * 2048, kQChunk, 1024),
                        sdesc_sw128(sa + kk * 2048, kQChunk, 1024), kQIdKV, (i > 0 || kk > 0));
            umma_commit(&sm.q_empty[hf]);
          }
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16(tmem + kColDv + hf * 64,
                        sdesc_sw128(da + hf * 2 * kQChunk + kk * 2048, kQChunk, 1024),
                        sdesc_sw128(pa + kk * 2048, kQChunk, 1024), kQIdKV, (i > 0 || kk > 0));
            umma_commit(&sm.do_empty[hf]);
          }
          umma_commit(&sm.pds_empty);
        }
        umma_commit(&sm.acc_full);
        ++ic;
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P, dS and epilogue
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int tok = r / kQG, hd = r - (r / kQG) * kQG;
    const uint32_t trow = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = scale * kQLog2e;
    uint32_t ic = 0, n = 0;
    bool ok = true;
    for (uint32_t wu = 0; ok; ++wu) {
      int jt = 0;
      if (lane == 0) jt = ring_get(sm.ring, wu, status, 62);
      jt = __shfl_sync(0xffffffffu, jt, 0);
      if (jt == kRingTimeout) ok = false;
      if (jt < 0) break;
      const int it = __ldg(ord + jt);
      const int* kl = klist + (static_cast<size_t>(it) * Hkv + g) * (1 + kQWin);
      const int nq = __ldg(kl);
      if (nq == 0) continue;
      const int4 item = items[it];
      const int seq0 = __ldg(cu + item.x), len = __ldg(cu + item.x + 1) - seq0;
      const int kt = item.y;
      for (int i = 0; i < nq; ++i, ++n) {
        const int qt = __ldg(kl + 1 + i);
        const int pos = qt * kQTok + tok;
        const bool valid = r < kQRows && pos < len;
        const size_t qrow = static_cast<size_t>(seq0 + pos) * Hq + g * kQG + hd;
        const uint32_t bits =
            valid ? tile_bits(masks + (static_cast<size_t>(seq0 + pos) * Hkv + g) * W, kt) : 0u;
        const float2 ld = valid ? __ldg(lsd + qrow) : make_float2(0.f, 0.f);
        const int kmax = pos - kt * kQKeys;
        if (!(ok = mbar_wait(&sm.s_full, n & 1, status, 49))) break;
        __syncwarp();
        tc_fence_after();
        uint32_t sv[64], dv[64];
        tmem_ld32(tmem + kColS + trow, sv);
        tmem_ld32(tmem + kColS + trow + 32, sv + 32);
        tmem_ld32(tmem + kColDp + trow, dv);
        tmem_ld32(tmem + kColDp + trow + 32, dv + 32);
        tmem_ld_wait();
        // P / dS of the previous query tile must have been consumed
        if (n > 0 && !(ok = mbar_wait(&sm.pds_empty, (n - 1) & 1, status, 50))) break;
        uint8_t* prow = sm.p;
        uint8_t* srow = sm.ds;
        // keys in pairs: both lie in one 4-key block, so one selection bit
        // serves the pair; fp32 math two lanes at a time
        const float2 sl2v = make_float2(sl2, sl2), lxv = make_float2(ld.x, ld.x),
                     lyv = make_float2(ld.y, ld.y);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t pw[4], sw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 8 * c + 2 * e;
            const bool blk = (bits >> (j >> 2)) & 1u;
            const float2 y = ffma2(make_float2(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])),
                                   sl2v, lxv);
            const float2 pe = make_float2(qex2(y.x), qex2(y.y));
            const float2 dd = fmul2(
                pe, fadd2(make_float2(__uint_as_float(dv[j]), __uint_as_float(dv[j + 1])), lyv));
            const bool k0 = blk && j <= kmax, k1 = blk && j + 1 <= kmax;
            pw[e] = pack_bf16x2(k0 ? pe.x : 0.f, k1 ? pe.y : 0.f);
            sw[e] = pack_bf16x2(k0 ? dd.x : 0.f, k1 ? dd.y : 0.f);
          }
          const uint32_t off = sw128_offset(static_cast<uint32_t>(r), static_cast<uint32_t>(c));
          *reinterpret_cast<uint4*>(prow + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          *reinterpret_cast<uint4*>(srow + off) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&sm.pds_full);
      }
      if (!ok) break;
      // ---- epilogue: lane r of half hf holds dimension 128 hf + r of 64 keys
      if (!(ok = mbar_wait(&sm.acc_full, ic & 1, status, 51))) break;
      __syncwarp();
      tc_fence_after();
      const int key0 = kt * kQKeys;
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        const int d = hf * 128 + r;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t a[32], b[32];
          tmem_ld32(tmem + kColDv + hf * 64 + trow + 32 * c, a);
          tmem_ld32(tmem + kColDk + hf * 64 + trow + 32 * c, b);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int key = key0 + 32 * c + j;
            if (key < len) {
              const size_t idx = (static_cast<size_t>(seq0 + key) * Hkv + g) * kQD + d;
              atomicAdd(dv_acc + idx, __uint_as_float(a[j]));
              atomicAdd(dk_acc + idx, __uint_as_float(b[j]) * scale);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.acc_free);
      ++ic;
    }
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// dk = bf16(dk_acc), dv = bf16(dv_acc); 8 elements per thread.
__global__ void __launch_bounds__(256) qsa_convert_kernel(const float* __restrict__ dk_acc,
                                                          const float* __restrict__ dv_acc,
                                                          __nv_bfloat16* __restrict__ dk,
                                                          __nv_bfloat16* __restrict__ dv,
                                                          size_t n8) {
  pdl_enter();
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < 2 * n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const bool is_v = i >= n8;
    const size_t e = is_v ? i - n8 : i;
    const float4* src = reinterpret_cast<const float4*>(is_v ? dv_acc : dk_acc) + 2 * e;
    const float4 a = __ldcs(src), b = __ldcs(src + 1);
    uint4 out;
    out.x = pack_bf16x2(a.x, a.y);
    out.y = pack_bf16x2(a.z, a.w);
    out.z = pack_bf16x2(b.x, b.y);
    out.w = pack_bf16x2(b.z, b.w);
    reinterpret_cast<uint4*>(is_v ? dv : dk)[e] = out;
  }
}

// ---------------------------------------------------------------- host side

#define QSA_TRY(expr)                 \
  do {                                \
    msa_status_t _e = (expr);         \
    if (_e != MSA_OK) return _e;      \
  } while (0)

int qsa_mask_words(int max_seqlen) { return (max_seqlen + 32 * kQBlk - 1) / (32 * kQBlk); }

static int qsa_ustride(int max_seqlen) { return 1 + (max_seqlen + kQKeys - 1) / kQKeys; }

static int qsa_max_items(int T, int S, int max_seqlen) {
  const int windows = ((max_seqlen + kQTok - 1) / kQTok + kQWin - 1) / kQWin;
  return (T / kQKeys + S) * windows;
}

static int capped_blocks(size_t work, int per_block, int cap) {
  const size_t b = (work + per_block - 1) / per_block;
  return static_cast<int>(b < static_cast<size_t>(cap) ? (b > 0 ? b : 1) : cap);
}

QsaFwdWorkspace carve_qsa_fwd_workspace(WsCursor& ws, int T, int S, int Hkv, int max_seqlen) {
  QsaFwdWorkspace w;
  w.plan = carve_plan(ws, T, S, kQTok);
  w.W = qsa_mask_words(max_seqlen);
  w.masks = ws.take<uint32_t>(static_cast<size_t>(T) * Hkv * w.W);
  w.ustride = qsa_ustride(max_seqlen);
  w.ulist = ws.take<int>(static_cast<size_t>(w.plan.max_tiles) * Hkv * w.ustride);
  w.tile_ctr = ws.take<int>(Hkv);
  return w;
}

QsaBwdWorkspace carve_qsa_bwd_workspace(WsCursor& ws, int T, int S, int Hq, int Hkv,
                                        int max_seqlen) {
  QsaBwdWorkspace w;
  w.map = carve_qsa_fwd_workspace(ws, T, S, Hkv, max_seqlen);
  w.lsd = ws.take<float2>(static_cast<size_t>(T) * Hq);
  w.max_items = qsa_max_items(T, S, max_seqlen);
  w.items = ws.take<int4>(w.max_items);
  w.num_items = ws.take<int>(1);
  w.klist = ws.take<int>(static_cast<size_t>(w.max_items) * Hkv * (1 + kQWin));
  w.order = ws.take<int>(static_cast<size_t>(w.max_items) * Hkv);
  w.num_busy = ws.take<int>(Hkv);
  w.item_ctr = ws.take<int>(Hkv);
  // the two accumulators stay adjacent: one clear covers them
  w.dk_acc = ws.take<float>(static_cast<size_t>(T) * Hkv * kQD);
  w.dv_acc = ws.take<float>(static_cast<size_t>(T) * Hkv * kQD);
  return w;
}

// masks, plan and tile map: shared by the forward and the backward
static msa_status_t launch_qsa_tilemap(const int32_t* sel, const int32_t* cu, int S, int T,
                                       int Hkv, int topk, int max_seqlen,
                                       const QsaFwdWorkspace& fw, cudaStream_t stream) {
  const int sms = device_sm_count();
  uint32_t* sw = nullptr;
  if (msa_status_t e_ = status_word(&sw); e_ != MSA_OK) return e_;
  {
    TraceScope trace_("qsa_mask_kernel", stream);
    launch_pdl(qsa_mask_kernel, capped_blocks(static_cast<size_t>(T) * Hkv, 8, 8 * sms), 256, 0,
        stream, sel, cu, S, T, Hkv, topk, fw.W, fw.masks,
        (topk % 4 == 0 && (reinterpret_cast<uintptr_t>(sel) & 15) == 0) ? 1 : 0, sw);
  }
  QSA_TRY(check_launch("qsa_mask_kernel"));
  QSA_TRY(launch_plan(fw.plan, cu, S, max_seqlen, stream));
  {
    TraceScope trace_("qsa_union_kernel", stream);
    launch_pdl(qsa_union_kernel,
        capped_blocks(static_cast<size_t>(fw.plan.max_tiles) * Hkv, 8, 4 * sms), 256, 0, stream,
        fw.masks, fw.W, cu, fw.plan.tiles, fw.plan.num_tiles, Hkv, fw.ustride, fw.ulist,
        fw.tile_ctr, sw);
  }
  return check_launch("qsa_union_kernel");
}

static bool qsa_maps(const void* q, const void* k, const void* v, const void* dout, int T,
                     int Hq, int Hkv, CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv,
                     CUtensorMap* tdo) {
  const uint64_t dq[3] = {static_cast<uint64_t>(kQD), static_cast<uint64_t>(Hq),
                          static_cast<uint64_t>(T)};
  const uint64_t dkv[3] = {static_cast<uint64_t>(kQD), static_cast<uint64_t>(Hkv),
                           static_cast<uint64_t>(T)};
  const uint32_t bq[3] = {64, static_cast<uint32_t>(kQG), static_cast<uint32_t>(kQTok)};
  const uint32_t bkv[3] = {64, 1, static_cast<uint32_t>(kQKeys)};
  return make_tmap_bf16(tq, q, 3, dq, bq) && make_tmap_bf16(tk, k, 3, dkv, bkv) &&
         make_tmap_bf16(tv, v, 3, dkv, bkv) && (!dout || make_tmap_bf16(tdo, dout, 3, dq, bq));
}

msa_status_t launch_qsa_fwd(const void* q, const void* k, const void* v, const int32_t* sel,
                            const int32_t* cu, int S, int T, int Hq, int Hkv, int topk,
                            int max_seqlen, float scale, const QsaFwdWorkspace& fw, void* o,
                            float* lse, cudaStream_t stream) {
  if (Hq != kQG * Hkv)
    return fail(MSA_ERR_UNSUPPORTED, "narrow-block attention needs Hq = 12 Hkv (got %d, %d)",
                Hq, Hkv);
  CUtensorMap tq, tk, tv;
  if (!qsa_maps(q, k, v, nullptr, T, Hq, Hkv, &tq, &tk, &tv, nullptr))
    return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the narrow-block q/k/v");
  uint32_t* sw = nullptr;
  if (msa_status_t e_ = status_word(&sw); e_ != MSA_OK) return e_;
  QSA_TRY(launch_qsa_tilemap(sel, cu, S, T, Hkv, topk, max_seqlen, fw, stream));
  const size_t smem = sizeof(QsaFwdSmem) + 1024;
  QSA_TRY(ensure_smem(qsa_fwd_kernel, smem, "qsa_fwd_kernel"));
  const int per_head = (device_sm_count() + Hkv - 1) / Hkv;
  dim3 grid(static_cast<unsigned>(per_head < fw.plan.max_tiles ? per_head : fw.plan.max_tiles),
            Hkv);
  {
    TraceScope trace_("qsa_fwd_kernel", stream);
    launch_pdl(qsa_fwd_kernel, grid, kQFwdThreads, smem, stream, tq, tk, tv, fw.masks, fw.W,
        fw.ulist, fw.ustride, cu, fw.plan.tiles, fw.plan.num_tiles, Hq, Hkv, scale,
        static_cast<__nv_bfloat16*>(o), lse, fw.tile_ctr, sw);
  }
  return check_launch("qsa_fwd_kernel");
}

msa_status_t launch_qsa_bwd(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, const int32_t* sel,
                            const int32_t* cu, int S, int T, int Hq, int Hkv, int topk,
                            int max_seqlen, float scale, const QsaBwdWorkspace& w, void* dq,
                            void* dk, void* dv, cudaStream_t stream) {
  if (Hq != kQG * Hkv)
    return fail(MSA_ERR_UNSUPPORTED, "narrow-block attention needs Hq = 12 Hkv (got %d, %d)",
                Hq, Hkv);
  CUtensorMap tq, tk, tv, tdo;
  if (!qsa_maps(q, k, v, dout, T, Hq, Hkv, &tq, &tk, &tv, &tdo))
    return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the narrow-block backward");
  uint32_t* sw = nullptr;
  if (msa_status_t e_ = status_word(&sw); e_ != MSA_OK) return e_;
  const int sms = device_sm_count();
  const QsaFwdWorkspace& fw = w.map;
  QSA_TRY(launch_qsa_tilemap(sel, cu, S, T, Hkv, topk, max_seqlen, fw, stream));

  const size_t nkv = static_cast<size_t>(T) * Hkv * kQD;
  if (w.dv_acc != w.dk_acc + nkv) return fail(MSA_ERR_CUDA, "dK/dV accumulators not adjacent");
  if (cudaMemsetAsync(w.dk_acc, 0, 2 * nkv * sizeof(float), stream) != cudaSuccess)
    return fail(MSA_ERR_CUDA, "workspace clear failed");
  const size_t rows = static_cast<size_t>(T) * Hq;
  {
    TraceScope trace_("qsa_delta_kernel", stream);
    launch_pdl(qsa_delta_kernel, capped_blocks(rows, 16, 16 * sms), 256, 0, stream,
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse,
        w.lsd, rows);
  }
  {
    TraceScope trace_("qsa_items_kernel", stream);
    launch_pdl(qsa_items_kernel, 1, 1024, 0, stream, cu, S, w.items, w.num_items, w.max_items,
        sw);
  }
  {
    TraceScope trace_("qsa_kvlist_kernel", stream);
    launch_pdl(qsa_kvlist_kernel, capped_blocks(static_cast<size_t>(w.max_items) * Hkv, 8, 4 * sms),
        256, 0, stream, fw.masks, fw.W, cu, w.items, w.num_items, Hkv, w.klist);
  }
  {
    TraceScope trace_("qsa_order_kernel", stream);
    launch_pdl(qsa_order_kernel, Hkv, 1024, 0, stream, w.klist, w.num_items, Hkv, w.max_items,
        w.order, w.num_busy, w.item_ctr);
  }
  QSA_TRY(check_launch("qsa_delta/items/kvlist/order"));

  const size_t smem_dq = sizeof(QsaDqSmem) + 1024;
  QSA_TRY(ensure_smem(qsa_bwd_dq_kernel, smem_dq, "qsa_bwd_dq_kernel"));
  const int per_head = (sms + Hkv - 1) / Hkv;
  {
    dim3 grid(static_cast<unsigned>(per_head < fw.plan.max_tiles ? per_head : fw.plan.max_tiles),
              Hkv);
    TraceScope trace_("qsa_bwd_dq_kernel", stream);
    launch_pdl(qsa_bwd_dq_kernel, grid, kQBwdThreads, smem_dq, stream, tq, tdo, tk, tv,
        fw.masks, fw.W, fw.ulist, fw.ustride, w.lsd, cu, fw.plan.tiles, fw.plan.num_tiles, Hq,
        Hkv, scale, static_cast<__nv_bfloat16*>(dq), w.map.tile_ctr, sw);
  }
  QSA_TRY(check_launch("qsa_bwd_dq_kernel"));

  const size_t smem_kv = sizeof(QsaDkvSmem) + 1024;
  QSA_TRY(ensure_smem(qsa_bwd_dkv_kernel, smem_kv, "qsa_bwd_dkv_kernel"));
  {
    dim3 grid(static_cast<unsigned>(per_head < w.max_items ? per_head : w.max_items), Hkv);
    TraceScope trace_("qsa_bwd_dkv_kernel", stream);
    launch_pdl(qsa_bwd_dkv_kernel, grid, kQBwdThreads, smem_kv, stream, tq, tdo, tk, tv,
        fw.masks, fw.W, w.klist, w.lsd, cu, w.items, w.order, w.num_busy, w.max_items, Hq, Hkv,
        scale, w.dk_acc, w.dv_acc, w.item_ctr, sw);
  }
  QSA_TRY(check_launch("qsa_bwd_dkv_kernel"));
  {
    TraceScope trace_("qsa_convert_kernel", stream);
    launch_pdl(qsa_convert_kernel, capped_blocks(nkv / 8 * 2, 256, 8 * sms), 256, 0, stream,
        w.dk_acc, w.dv_acc, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv),
        nkv / 8);
  }
  return check_launch("qsa_convert_kernel");
}

}  // namespace msa
