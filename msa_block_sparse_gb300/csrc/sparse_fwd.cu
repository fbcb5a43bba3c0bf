// Block-sparse GQA attention forward ("MiniMax-M3.1-Flash", 1 "Model
// Introduction": each query attends to its 16 selected 128-token blocks, own
// block included, causally; "#4581", "Kernel tuning": QSA block-sparse kernel).
//
// Tile = 128 rows = 8 consecutive tokens x the 16 query heads of one KV head, so
// a single K/V block feeds every row.  The tile's tokens lie in one 128-token
// block and share their own block.  The tile walks the union of its tokens'
// selected blocks in ascending order; a row whose token did not select the
// current block gets P = 0 for it.
//
// Persistent CTAs (one per SM) claim tiles from a counter:
//   producers: warp 0 claims the next tile, copies its block union (built
//            beforehand by fwd_union_kernel, one warp per tile) into a
//            double-buffered slot, loads its Q tile and streams K_b through a
//            2-stage TMA ring; warp 10 streams V_b through its own 2-stage
//            ring, so neither ring's release holds up the other
//   MMA (warps 1 and 11, one per 64-key half h): S_h = Q K_b[64h, 64h+64)^T
//            into one of two TMEM buffers of the half; then
//            O_h += P_h V_b[64h, 64h+64) with P_h read from TMEM as the A operand
//   softmax (warps 2..9): warp = 32 rows x one 64-key half h.  Each half keeps
//            its own running max (log2 domain, rescaled only when it grows by
//            more than 2^8, so P < 256 fits bf16), row sum and O_h accumulator;
//            P_h is packed to bf16 into the S buffer it came from.  The
//            epilogue merges the halves, o = (O_0 2^(m_0-m) + O_1 2^(m_1-m)) / l,
//            stages a full tile in its (finished) Q buffer and writes it with
//            one tensor store per half; the next tile's first PV waits until
//            both halves have read O_0 and O_1.
#include "kernels.cuh"

namespace msa {

namespace {

// warp 0 Q/K producer, warps 1 and 11 MMA (key half 0 / 1), warps 2..9
// softmax, warp 10 V producer
constexpr int kFwdThreads = 384;
constexpr int kVLoaderWarp = 10;
constexpr int kMmaWarp1 = 11;

constexpr int kSoftmaxThreads = 256;
constexpr int kHalfThreads = kSoftmaxThreads / 2;   // softmax threads of one key half
constexpr int kFirstHalfWarp = 2;           // warps 2..5: key half 0, 6..9: key half 1
constexpr int kG = 16;                      // query heads per KV head
constexpr int kTpt = 8;                     // tokens per tile
constexpr int kTile = 128 * 128 * 2;        // bytes of a 128 x 128 bf16 tile
constexpr int kHalf = kTile / 2;            // one 64-column half
constexpr int kMaskWords = kMaxSeqlen / kBlock / 32;
constexpr uint32_t kIdescS = idesc_bf16(128, 64, false, false);    // S_h: 64 keys of a half
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, false, true);   // O_h += P_h V_h
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 of the largest P before a rescale
constexpr uint32_t kColO = 256;             // O_0 at 256, O_1 at 384; S buffers at 0, 128

struct TileInfo {
  int s, qb, seq0, len, p0, ntok;
};

struct FwdSmem {
  uint8_t q[2][kTile];
  uint8_t k[2][kTile];
  uint8_t v[2][kTile];
  int ublk[2][kTpt * kTopK];                 // union entries (block << 8) | token mask
  int n_union[2];
  int tile_id[2];                           // tile of the slot; -1: no tiles left
  TileInfo tinfo[2];                        // its decoded plan entry (read once, by warp 0)
  float2 ml[2][128];                        // per half: (max, sum) of each row, for the merge
  uint64_t tile_full[2], tile_empty[2];
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  // per key half and S buffer: a waiter is then never more than one phase behind
  uint64_t s_full[2][2], p_full[2][2], pv_done[2][2], ml_full;
  uint64_t o_done[2];                       // a half's threads have read O and staged their rows
  uint64_t o_free;                          // both halves have read O_0 and O_1 of the tile
  uint32_t tmem_base;
};
static_assert(sizeof(FwdSmem) <= 232448, "forward shared memory above the 227 KB limit");

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



// Global tile ti -> plan tile ti / 16 (a 128-token block), sub-tile ti % 16.
__device__ __forceinline__ bool tile_info(int ti, const int2* tiles, const int32_t* cu,
                                          TileInfo& t) {
  const int2 pt = tiles[ti >> 4];
  t.s = pt.x;
  t.qb = pt.y;
  t.seq0 = cu[t.s];
  t.len = cu[t.s + 1] - t.seq0;
  t.p0 = t.qb * kBlock + (ti & 15) * kTpt;
  t.ntok = min(kTpt, t.len - t.p0);
  return t.p0 < t.len;
}

}  // namespace

// One warp per (tile, KV head), grid-striding: the union of the 8 tokens'
// selected blocks in ascending order, each entry (block << 8) | token mask.
__global__ void __launch_bounds__(256) fwd_union_kernel(const int32_t* __restrict__ sel,
                                                        const int32_t* __restrict__ cu,
                                                        const int2* __restrict__ tiles,
                                                        const int* __restrict__ num_tiles,
                                                        int Hkv, int* __restrict__ ulist,
                                                        int* __restrict__ tile_ctr,
                                                        uint32_t* status) {
  pdl_enter();
  __shared__ uint32_t words_s[8][kMaskWords];
  const int total = *num_tiles * kG;
  const int g = blockIdx.y;
  if (blockIdx.x == 0 && threadIdx.x == 0) tile_ctr[g] = 0;   // the forward claims from 0
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int ti = blockIdx.x * 8 + warp; ti < total; ti += gridDim.x * 8) {
    int* out = ulist + (static_cast<size_t>(ti) * Hkv + g) * kFwdUnionStride;
    TileInfo t;
    if (!tile_info(ti, tiles, cu, t)) {
      if (lane == 0) out[0] = 0;
      continue;
    }
    int ids[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = lane * 4 + e;             // lanes 4i .. 4i+3 hold token i's 16 ids
      const int tl = idx >> 4;
      int b = -1;
      if (tl < t.ntok) {
        b = __ldg(sel + (static_cast<size_t>(t.seq0 + t.p0 + tl) * Hkv + g) * kTopK + (idx & 15));
        if (b > t.qb) {
          atomicOr(status, kStatusBounds);
          b = -1;
        }
      }
      ids[e] = b;
    }
    const int nb_seq = (t.len + kBlock - 1) / kBlock;
    const int words = min((nb_seq + 31) >> 5, kMaskWords);
    if (lane < words) words_s[warp][lane] = 0;
    __syncwarp();
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (ids[e] >= 0) atomicOr(&words_s[warp][ids[e] >> 5], 1u << (ids[e] & 31));
    __syncwarp();
    int n = 0;
    for (int w = 0; w < words; ++w) {
      uint32_t u = words_s[warp][w];
      while (u) {
        const int b = w * 32 + __ffs(u) - 1;
        u &= u - 1;
        const bool mine = (ids[0] == b) | (ids[1] == b) | (ids[2] == b) | (ids[3] == b);
        const uint32_t bal = __ballot_sync(0xffffffffu, mine);
        uint32_t tm = 0;
#pragma unroll
        for (int i = 0; i < kTpt; ++i) tm |= ((bal >> (4 * i)) & 0xFu) ? (1u << i) : 0u;
        if (lane == 0 && n < kTpt * kTopK) out[4 + n] = (b << 8) | static_cast<int>(tm);
        ++n;
      }
    }
    if (lane == 0) out[0] = min(n, kTpt * kTopK);
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kFwdThreads, 1)
    sparse_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, const int* __restrict__ ulist,
                      int* __restrict__ tile_ctr, const int32_t* __restrict__ cu, const int2* __restrict__ tiles,
                      const int* __restrict__ num_tiles, int Hq, int Hkv, float scale,
                      __nv_bfloat16* __restrict__ o, float* __restrict__ lse, uint32_t* status) {
  pdl_enter();
  const int total = *num_tiles * kG;
  if (static_cast<int>(blockIdx.x) >= total) return;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {   // the tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(status, kStatusBounds);
    return;
  }
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(smem_raw);
  const int g = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.tile_full[i], 1);
      mbar_init(&sm.tile_empty[i], 2 + 2 + 1);
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 2);
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 2);
      for (int hh = 0; hh < 2; ++hh) {
        mbar_init(&sm.s_full[hh][i], 1);
        mbar_init(&sm.p_full[hh][i], kHalfThreads);
        mbar_init(&sm.pv_done[hh][i], 1);
      }
    }
    mbar_init(&sm.ml_full, kSoftmaxThreads);
    mbar_init(&sm.o_free, 2);
    mbar_init(&sm.o_done[0], kHalfThreads);
    mbar_init(&sm.o_done[1], kHalfThreads);
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
      prefetch_tmap(&tm_k);
    }
    // Tiles are claimed from a per-KV-head counter (heaviest first, as the plan
    // orders them) so that CTAs finishing early take more; the claimed id goes
    // to the other roles through the tile slot, -1 once none are left.
    uint32_t tcount = 0, kc = 0;
    bool alive = true;
    int pending = 0;
    if (lane == 0) pending = atomicAdd(tile_ctr + g, 1);
    while (alive) {
      int ti = -1;
      if (lane == 0) {
        ti = pending;
        TileInfo tt;
        while (ti < total && !tile_info(ti, tiles, cu, tt)) ti = atomicAdd(tile_ctr + g, 1);
        if (ti >= total) ti = -1;
      }
      ti = __shfl_sync(0xffffffffu, ti, 0);
      const int tb = tcount & 1;
      if (lane == 0) alive = mbar_wait(&sm.tile_empty[tb], ((tcount >> 1) & 1) ^ 1, status, 1);
      alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
      if (!alive) break;
      if (ti < 0) {
        if (lane == 0) {
          sm.tile_id[tb] = -1;
          mbar_arrive(&sm.tile_full[tb]);
        }
        break;
      }
      TileInfo t;
      tile_info(ti, tiles, cu, t);
      // ---- the tile's union entries (built by fwd_union_kernel)
      const int* ul = ulist + (static_cast<size_t>(ti) * Hkv + g) * kFwdUnionStride;
      const int nU = min(__ldg(ul), kTpt * kTopK);
      for (int i = lane; i < nU; i += 32) sm.ublk[tb][i] = __ldg(ul + 4 + i);
      if (lane == 0) {
        sm.n_union[tb] = nU;
        sm.tile_id[tb] = ti;
        sm.tinfo[tb] = t;
      }
      __syncwarp();
      if (lane == 0) {
        pending = atomicAdd(tile_ctr + g, 1);   // next claim, in flight while K streams
        mbar_arrive_expect_tx(&sm.tile_full[tb], kTile);
        tma_load_3d(sm.q[tb], &tm_q, &sm.tile_full[tb], 0, g * kG, t.seq0 + t.p0);
        tma_load_3d(sm.q[tb] + kHalf, &tm_q, &sm.tile_full[tb], 64, g * kG, t.seq0 + t.p0);
        // ---- K tiles through their 2-stage ring (V has its own warp, so a V
        // slot that frees late does not hold up the next K)
        for (int i = 0; alive && i < nU; ++i) {
          const int st = kc & 1;
          if (!(alive = mbar_wait(&sm.k_empty[st], ((kc >> 1) & 1) ^ 1, status, 2))) break;
          const int row = t.seq0 + (sm.ublk[tb][i] >> 8) * kBlock;
          mbar_arrive_expect_tx(&sm.k_full[st], kTile);
          tma_load_3d(sm.k[st], &tm_k, &sm.k_full[st], 0, g, row);
          tma_load_3d(sm.k[st] + kHalf, &tm_k, &sm.k_full[st], 64, g, row);
          ++kc;
        }
      }
      alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
      ++tcount;
    }
  } else if (warp == kVLoaderWarp) {
    // ------------------------------------------------------------ V producer
    if (lane == 0) {
      prefetch_tmap(&tm_v);
      uint32_t tcount = 0, vc = 0;
      bool alive = true;
      for (;;) {
        const int tb = tcount & 1;
        // the tile's union list is in place once its Q has landed
        if (!(alive = mbar_wait(&sm.tile_full[tb], (tcount >> 1) & 1, status, 15))) break;
        if (sm.tile_id[tb] < 0) break;
        const TileInfo t = sm.tinfo[tb];
        const int nU = sm.n_union[tb];
        for (int i = 0; alive && i < nU; ++i) {
          const int st = vc & 1;
          if (!(alive = mbar_wait(&sm.v_empty[st], ((vc >> 1) & 1) ^ 1, status, 3))) break;
          const int row = t.seq0 + (sm.ublk[tb][i] >> 8) * kBlock;
          mbar_arrive_expect_tx(&sm.v_full[st], kTile);
          tma_load_3d(sm.v[st], &tm_v, &sm.v_full[st], 0, g, row);
          tma_load_3d(sm.v[st] + kHalf, &tm_v, &sm.v_full[st], 64, g, row);
          ++vc;
        }
        if (!alive) break;
        mbar_arrive(&sm.tile_empty[tb]);   // done reading the tile's union list
        ++tcount;
      }
    }
  } else if (warp == 1 || warp == kMmaWarp1) {
    // ------------------------------------------------------------ MMA issuers
    // one per key half hh: S_hh = Q K[64hh, 64hh+64)^T and O_hh += P_hh V[64hh, ..)
    const int hh = (warp == 1) ? 0 : 1;
    if (elect_one()) {
      uint32_t tcount = 0, kc = 0, vc = 0, bc = 0;
      bool ok = true;
      for (;;) {
        const int tb = tcount & 1;
        if (!(ok = mbar_wait(&sm.tile_full[tb], (tcount >> 1) & 1, status, 4))) break;
        if (sm.tile_id[tb] < 0) break;
        tc_fence_after();
        const int nU = sm.n_union[tb];
        const uint32_t qa = smem_u32(sm.q[tb]);
        const uint32_t bc0 = bc;
        for (int i = 0; ok && i <= nU; ++i) {
          if (i < nU) {
            const int st = kc & 1;
            if (!(ok = mbar_wait(&sm.k_full[st], (kc >> 1) & 1, status, 5))) break;
            // this half of S buffer bc held P of block bc - 2: wait for its PV
            if (bc >= 2 &&
                !(ok = mbar_wait(&sm.pv_done[hh][bc & 1], ((bc - 2) >> 1) & 1, status, 6)))
              break;
            tc_fence_after();
            // keys [64hh, 64hh + 64) of the K tile: rows 64hh.. of both D halves
            const uint32_t ka = smem_u32(sm.k[st]) + hh * 64 * 128;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
              umma_bf16(tmem + (bc & 1) * 128 + 64 * hh, sdesc_sw128(qa + off, 16, 1024),
                        sdesc_sw128(ka + off, 16, 1024), kIdescS, kk > 0);
            }
            umma_commit(&sm.s_full[hh][bc & 1]);
            umma_commit(&sm.k_empty[st]);
            ++kc;
            ++bc;
          }
          if (i > 0) {
            const uint32_t j = bc0 + i - 1;
            const int st = vc & 1;
            if (!(ok = mbar_wait(&sm.p_full[hh][j & 1], (j >> 1) & 1, status, 7))) break;
            if (!(ok = mbar_wait(&sm.v_full[st], (vc >> 1) & 1, status, 8))) break;
            // the tile's first PV overwrites O_hh: the previous tile's epilogue
            // (both halves) must have read it
            if (i == 1 && tcount > 0 &&
                !(ok = mbar_wait(&sm.o_free, (tcount - 1) & 1, status, 16)))
              break;
            tc_fence_after();
            // V rows (keys) [64hh, 64hh + 64): four K-steps of 16 keys
            const uint32_t va = smem_u32(sm.v[st]) + hh * 64 * 128;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t a_t = tmem + (j & 1) * 128 + hh * 64 + kk * 8;
              umma_bf16_tmem_a(tmem + kColO + hh * 128, a_t,
                               sdesc_sw128(va + kk * 2048, kHalf, 1024), kIdescPV,
                               (i > 1 || kk > 0));
            }
            umma_commit(&sm.pv_done[hh][j & 1]);
            umma_commit(&sm.v_empty[st]);
            ++vc;
          }
        }
        if (!ok) break;
        umma_commit(&sm.tile_empty[tb]);   // Q of this tile is free once its S MMAs are done
        ++tcount;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int cw = warp - 2;
    const int subp = warp & 3;
    const int h = cw >> 2;                   // key half [64h, 64h + 64) of every block
    const int r = subp * 32 + lane;          // tile row = TMEM lane
    const int tl = r >> 4, hd = r & 15;      // token of the tile, head of the group
    const uint32_t trow = static_cast<uint32_t>(subp * 32) << 16;
    const float sl2 = scale * kLog2e;
    uint32_t tcount = 0, bc = 0;
    bool ok = true;
    for (;;) {
      const int tb = tcount & 1;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&sm.tile_full[tb], (tcount >> 1) & 1, status, 9))))
        break;
      if (sm.tile_id[tb] < 0) break;
      const TileInfo t = sm.tinfo[tb];
      const int nU = sm.n_union[tb];
      const bool row_valid = tl < t.ntok;
      const int pos = t.p0 + tl;
      float m = -INFINITY, l = 0.f;
      for (int i = 0; i < nU; ++i) {
        const int ent = sm.ublk[tb][i];
        const int b = ent >> 8;
        const uint32_t sbuf = tmem + (bc & 1) * 128 + trow + 64 * h;
        if (!(ok = mbar_wait(&sm.s_full[h][bc & 1], (bc >> 1) & 1, status, 10))) break;
        __syncwarp();
        tc_fence_after();
        uint32_t sv[64];
        tmem_ld32(sbuf, sv);
        tmem_ld32(sbuf + 32, sv + 32);
        tmem_ld_wait();
        const bool selected = row_valid && ((ent >> tl) & 1);
        const int kmax = (b == t.qb) ? (pos & (kBlock - 1)) - 64 * h : 63;
        bool resc = false;
        float mu = m, rs = 0.f;
        uint32_t pk[32];
        if (selected && kmax >= 0) {
          float x[64];
#pragma unroll
          for (int j = 0; j < 64; ++j) x[j] = __uint_as_float(sv[j]);
          if (kmax < 63) {                    // own block: keys after the query are masked
#pragma unroll
            for (int j = 0; j < 64; ++j) x[j] = (j <= kmax) ? x[j] : -INFINITY;
          }
          // row max: eight independent chains of three-input maxima
          float mx8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float* xi = x + 8 * i;
            mx8[i] = fmaxf(max3f(max3f(max3f(xi[0], xi[1], xi[2]), xi[3], xi[4]), xi[5], xi[6]),
                           xi[7]);
          }
          const float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]),
                                 fmaxf(mx8[6], mx8[7]));
          const float mnew = fmaxf(m, mx * sl2);
          resc = mnew > m + kRescaleThreshold;
          mu = resc ? mnew : m;
          // p = exp2(s scale log2e - mu), two lanes of fp32 per instruction
          const float2 sl2v = make_float2(sl2, sl2), nmu = make_float2(-mu, -mu);
          float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                           make_float2(0.f, 0.f)};
#pragma unroll
          for (int j2 = 0; j2 < 32; ++j2) {
            const float2 y = ffma2(make_float2(x[2 * j2], x[2 * j2 + 1]), sl2v, nmu);
            const float2 pe = make_float2(ex2(y.x), ex2(y.y));
            acc[j2 & 3] = fadd2(acc[j2 & 3], pe);
            pk[j2] = pack_bf16x2(pe.x, pe.y);
          }
          const float2 a01 = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
          rs = a01.x + a01.y;
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) pk[j] = 0u;
        }
        const bool need = resc && m != -INFINITY;
        if (__any_sync(0xffffffffu, need)) {
          // O_h is stable only once the PV of the previous block is done
          if (!(ok = mbar_wait(&sm.pv_done[h][(bc - 1) & 1], ((bc - 1) >> 1) & 1, status, 11)))
            break;
          __syncwarp();
          tc_fence_after();
          const float alpha = need ? ex2(m - mu) : 1.f;
          const uint32_t orow = tmem + kColO + h * 128 + trow;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tmem_ld32(orow + c * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
            tmem_st16(orow + c * 32, v);
            tmem_st16(orow + c * 32 + 16, v + 16);
          }
        }
        if (selected && kmax >= 0) {
          l = (m == -INFINITY) ? rs : (resc ? l * ex2(m - mu) : l) + rs;
          m = mu;
        }
        tmem_st16(sbuf, pk);
        tmem_st16(sbuf + 16, pk + 16);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full[h][bc & 1]);
        ++bc;
      }
      if (!ok) break;
      // ---- epilogue: merge the two halves of every row
      // the PV of the tile's last block completes after all earlier ones
      if (!(ok = mbar_wait(&sm.pv_done[h][(bc - 1) & 1], ((bc - 1) >> 1) & 1, status, 13))) break;
      sm.ml[h][r] = make_float2(m, l);
      mbar_arrive(&sm.ml_full);
      if (!(ok = mbar_wait(&sm.ml_full, tcount & 1, status, 14))) break;
      const float2 other = sm.ml[h ^ 1][r];
      __syncwarp();
      tc_fence_after();
      const float M = fmaxf(m, other.x);
      const float f_me = (m == -INFINITY) ? 0.f : ex2(m - M);
      const float f_ot = (other.x == -INFINITY) ? 0.f : ex2(other.x - M);
      const float L = l * f_me + other.y * f_ot;
      const float f0 = (h == 0) ? f_me : f_ot, f1 = (h == 0) ? f_ot : f_me;
      const float inv = (L > 0.f) ? 1.f / L : 0.f;
      const size_t orow_g = static_cast<size_t>(t.seq0 + pos) * Hq + g * kG + hd;
      // A full tile is staged in its Q buffer (free: every MMA of the tile is
      // done) in the 128B-swizzled layout of the tensor map and written by one
      // tensor store per half; a partial tile (the end of a sequence) is
      // written row by row so that no row of the next sequence is touched.
      const bool full = t.ntok == kTpt;
      uint8_t* stage = sm.q[tb] + h * kHalf;
      uint4* dst = reinterpret_cast<uint4*>(o + orow_g * kD + 64 * h);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t a[32], bq[32];
        tmem_ld32(tmem + kColO + trow + 64 * h + 32 * c, a);
        tmem_ld32(tmem + kColO + 128 + trow + 64 * h + 32 * c, bq);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            x[e] = (__uint_as_float(a[8 * q + e]) * f0 + __uint_as_float(bq[8 * q + e]) * f1) * inv;
          uint4 pk;
          pk.x = pack_bf16x2(x[0], x[1]);
          pk.y = pack_bf16x2(x[2], x[3]);
          pk.z = pack_bf16x2(x[4], x[5]);
          pk.w = pack_bf16x2(x[6], x[7]);
          if (full)
            *reinterpret_cast<uint4*>(stage + sw128_offset(r, 4 * c + q)) = pk;
          else if (row_valid)
            dst[4 * c + q] = pk;
        }
      }
      tc_fence_before();
      if (full) fence_proxy_async_smem();      // staged rows -> the tensor store's reads
      mbar_arrive(&sm.o_done[h]);
      if (subp == kFirstHalfWarp % 4 && lane == 0) {
        // one thread per half: once all its rows are read and staged, release
        // O, store the staged half and hand the Q buffer back to the producer
        ok = mbar_wait(&sm.o_done[h], tcount & 1, status, 17);
        if (ok) {
          mbar_arrive(&sm.o_free);
          if (full) {
            tma_store_3d(&tm_o, stage, 64 * h, g * kG, t.seq0 + t.p0);
            bulk_commit_group();
            bulk_wait_read_all();             // the Q buffer may be reloaded after this
          }
          mbar_arrive(&sm.tile_empty[tb]);
        }
      }
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      if (h == 0 && row_valid) lse[orow_g] = (M + __log2f(L)) * 0.6931471805599453f;
      tc_fence_before();
      ++tcount;
    }
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

msa_status_t launch_sparse_fwd(const void* q, const void* k, const void* v, const int32_t* sel,
                               const int32_t* cu, int S, int T, int Hq, int Hkv, int max_seqlen,
                               float scale, const FwdWorkspace& fw, void* o, float* lse,
                               cudaStream_t stream) {
  const Plan& plan = fw.plan;
  (void)S;
  (void)max_seqlen;
  if (Hq / Hkv != kG)
    return fail(MSA_ERR_UNSUPPORTED, "forward supports Hq/Hkv = 16 (got %d)", Hq / Hkv);
  CUtensorMap tq, tk, tv, to;
  const uint64_t dq[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hq),
                          static_cast<uint64_t>(T)};
  const uint64_t dkv[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hkv),
                           static_cast<uint64_t>(T)};
  const uint32_t bq[3] = {64, static_cast<uint32_t>(kG), static_cast<uint32_t>(kTpt)};
  const uint32_t bkv[3] = {64, 1, 128};
  // o has q's layout: the same box stores one half of a tile's output
  if (!make_tmap_bf16(&tq, q, 3, dq, bq) || !make_tmap_bf16(&tk, k, 3, dkv, bkv) ||
      !make_tmap_bf16(&tv, v, 3, dkv, bkv) || !make_tmap_bf16(&to, o, 3, dq, bq))
    return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled failed for q/k/v/o");
  const size_t smem = sizeof(FwdSmem);
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(sparse_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    attr_set = true;
  }
  const int per_head = (device_sm_count() + Hkv - 1) / Hkv;
  const int max_ctas = plan.max_tiles * kG;
  dim3 grid(static_cast<unsigned>(per_head < max_ctas ? per_head : max_ctas), Hkv);
  {
    const int max_tiles16 = plan.max_tiles * kG;
    const int ublocks = (max_tiles16 + 7) / 8;
    const int cap = 4 * device_sm_count();
    dim3 ugrid(static_cast<unsigned>(ublocks < cap ? ublocks : cap), Hkv);
    TraceScope trace_("fwd_union_kernel", stream);
    launch_pdl(fwd_union_kernel, ugrid, 256, 0, stream, sel, cu, plan.tiles, plan.num_tiles, Hkv,
        fw.ulist, fw.tile_ctr, status_word());
  }
  {
    TraceScope trace_("sparse_fwd_kernel", stream);
    launch_pdl(sparse_fwd_kernel, grid, kFwdThreads, smem, stream,
        tq, tk, tv, to, fw.ulist, fw.tile_ctr, cu, plan.tiles, plan.num_tiles, Hq, Hkv, scale,
        static_cast<__nv_bfloat16*>(o), lse, status_word());
  }
  return check_launch("sparse_fwd_kernel");
}

FwdWorkspace carve_fwd_workspace(WsCursor& ws, int T, int S, int Hkv) {
  FwdWorkspace w;
  w.plan = carve_plan(ws, T, S);
  w.ulist = ws.take<int>(static_cast<size_t>(w.plan.max_tiles) * kG * Hkv * kFwdUnionStride);
  w.tile_ctr = ws.take<int>(Hkv);
  return w;
}

}  // namespace msa
