// Block-sparse GQA attention forward ("MiniMax-M3.1-Flash", 1 "Model
// Introduction": each query attends to its 16 selected 128-token blocks, own
// block included, causally; "#4581", "Kernel tuning": QSA block-sparse kernel).
//
// Tile = 128 rows = 8 tokens x the 16 query heads of one KV head, so a single
// K/V block feeds every row.  The tile's tokens lie in one 128-token query
// block (they share their own block) and are grouped there by selection
// similarity (fwd_union_kernel), so that the union of their selected blocks,
// which the tile walks in ascending order, stays small; a row whose token did
// not select the current block gets P = 0 for it.
//
// Persistent CTAs (one per SM) claim tiles from a counter:
//   producers: warp 0 claims the next tile, copies its block union (built
//            beforehand by fwd_union_kernel, one warp per tile) into a
//            double-buffered slot, loads its Q tile and streams K_b through a
//            2-stage TMA ring; warp 10 streams V_b through its own 2-stage
//            ring, so neither ring's release holds up the other, and for the
//            training forward zeroes a given region (the backward's fp32
//            accumulators) by 16 KB bulk copies of a zeroed shared buffer,
//            one after each V block, with the memory bandwidth the forward
//            leaves idle
//   MMA (warps 1 and 11, one per 64-key half h): S_h = Q K_b[64h, 64h+64)^T
//            into one of two TMEM buffers of the half; then
//            O_h += P_h V_b[64h, 64h+64) with P_h read from TMEM as the A operand
//   softmax (warps 2..9): warp = 32 rows x one 64-key half h.  Each half keeps
//            its own running max (log2 domain, rescaled only when it grows by
//            more than 2^8, so P < 256 fits bf16), row sum and O_h accumulator;
//            P_h is packed to bf16 into the S buffer it came from.  The
//            epilogue merges the halves, o = (O_0 2^(m_0-m) + O_1 2^(m_1-m)) / l,
//            stages the tile in its (finished) Q buffer and writes it with one
//            tensor store per token and half, each warp storing the two tokens
//            whose rows it holds; the next tile's first PV waits until both
//            halves have read O_0 and O_1.
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
constexpr int kTokRows = kG * 128;          // one token's 16 rows of a 64-column half
constexpr uint32_t kIdescS = idesc_bf16(128, 64, false, false);    // S_h: 64 keys of a half
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, false, true);   // O_h += P_h V_h
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 of the largest P before a rescale
constexpr uint32_t kColO = 256;             // O_0 at 256, O_1 at 384; S buffers at 0, 128

struct TileInfo {
  int s, qb, seq0, len, p0, ntok;   // p0: first position of the 128-token query block
  uint32_t offs[2];                 // byte i: offset in the block of the tile's i-th token
};

constexpr int kZeroBytes = 16384;          // zeroed source of the bulk clearing copies

struct FwdSmem {
  uint8_t q[2][kTile];
  uint8_t k[2][kTile];
  uint8_t v[2][kTile];
  alignas(16) uint8_t zero[kZeroBytes];
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



// Global tile ti -> plan tile ti / 16 (a 128-token query block), sub-tile
// (token group) ti % 16 of up to 8 of its tokens; the members are chosen by
// fwd_union_kernel and listed in the tile's union header.
__device__ __forceinline__ bool tile_info(int ti, const int2* tiles, const int32_t* cu,
                                          TileInfo& t) {
  const int2 pt = tiles[ti >> 4];
  t.s = pt.x;
  t.qb = pt.y;
  t.seq0 = cu[t.s];
  t.len = cu[t.s + 1] - t.seq0;
  t.p0 = t.qb * kBlock;
  const int first = (ti & 15) * kTpt;
  t.ntok = min(kTpt, t.len - t.p0 - first);
  t.offs[0] = t.offs[1] = 0;
  return t.p0 + first < t.len;
}

__device__ __forceinline__ int member_offset(const TileInfo& t, int i) {
  const uint32_t w = (i < 4) ? t.offs[0] : t.offs[1];
  return static_cast<int>((w >> (8 * (i & 3))) & 0xFFu);
}

// Token masks held in registers by the grouping: blocks below 32 x kGroupWords
// (query blocks of sequences up to 16,384 tokens); longer ones group
// consecutive tokens.
constexpr int kGroupWords = 4;

// Appends the union list of one token group: the blocks below the own block
// that any member selected (ascending, from the members' masks mm), each
// (block << 8) | member mask, then the own block (selected by every member).
__device__ __forceinline__ void write_union(int* out, const uint32_t (&mm)[kTpt][kGroupWords],
                                            int nm, int words, int qb, int lane) {
  int n = 0;
#pragma unroll
  for (int w = 0; w < kGroupWords; ++w) {
    if (w >= words) break;
    uint32_t tm = 0;
#pragma unroll
    for (int i = 0; i < kTpt; ++i) tm |= ((mm[i][w] >> lane) & 1u) << i;
    const uint32_t bal = __ballot_sync(0xffffffffu, tm != 0u);
    if (tm) out[4 + n + __popc(bal & ((1u << lane) - 1u))] = ((32 * w + lane) << 8) | tm;
    n += __popc(bal);
  }
  if (lane == 0) {
    out[4 + n] = (qb << 8) | ((1 << nm) - 1);
    out[0] = n + 1;
  }
}

}  // namespace

// One CTA per (128-token query block, KV head), grid-striding, of kWarps
// warps: warp w groups the block's tokens [w 128 / kWarps, (w + 1) 128 / kWarps)
// into tiles (sub-tiles 16 w / kWarps ..) of up to 8 tokens (the tile's MMA rows
// are 8 tokens x 16 heads) so that each tile's union of selected blocks - what
// its MMAs walk - stays small: a group starts from the lowest ungrouped token
// and repeatedly takes the token that adds the fewest blocks to the group's
// union (ties: the lower token).  Two warps (64 tokens each) halve the serial
// chain of greedy steps; one warp over all 128 tokens groups better, which pays
// on long sequences.  Per tile the header holds the member offsets and count,
// then the union in ascending order, each entry (block << 8) | member mask.
template <int kWarps>
__global__ void __launch_bounds__(32 * kWarps) fwd_union_kernel(const int32_t* __restrict__ sel,
                                                                  const int32_t* __restrict__ cu,
                                                                  const int2* __restrict__ tiles,
                                                                  const int* __restrict__ num_tiles,
                                                                  int Hkv, int* __restrict__ ulist,
                                                                  int* __restrict__ tile_ctr,
                                                                  uint32_t* status) {
  pdl_enter();
  constexpr int kWTok = kBlock / kWarps;         // tokens of one warp
  constexpr int kPerLane = kWTok / 32;
  __shared__ uint4 tok_mask[kWarps][kWTok];      // per warp: its tokens' masks (kGroupWords = 4)
  static_assert(kGroupWords == 4, "one uint4 per token mask");
  const int nblk = *num_tiles;
  const int g = blockIdx.y;
  if (blockIdx.x == 0 && threadIdx.x == 0) tile_ctr[g] = 0;   // the forward claims from 0
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int pb = blockIdx.x; pb < nblk; pb += gridDim.x) {
    const int2 pt = tiles[pb];
    const int qb = pt.y;
    const int seq0 = cu[pt.x];
    const int n = min(kBlock, cu[pt.x + 1] - seq0 - qb * kBlock);   // tokens of the block
    const int t0 = kWTok * warp;                                    // this warp's first token
    const int nw = max(0, min(kWTok, n - t0));                       // and its token count
    const int ngrp = (nw + kTpt - 1) / kTpt;
    auto tile_out = [&](int grp) {
      return ulist + (static_cast<size_t>(pb * kG + (kG / kWarps) * warp + grp) * Hkv + g) *
                         kFwdUnionStride;
    };
    if (lane >= ngrp && lane < kG / kWarps) tile_out(lane)[0] = 0;
    const bool fits = qb < 32 * kGroupWords;
    const int words = fits ? (qb + 31) / 32 : 0;
    // ---- the tokens' masks of selected earlier blocks (own block left out);
    // all loads first, then the bits
    int4 ids[kPerLane][4];
#pragma unroll
    for (int k = 0; k < kPerLane; ++k) {
      const int tok = t0 + lane + 32 * k;
      const int4* row = reinterpret_cast<const int4*>(
          sel + (static_cast<size_t>(seq0 + qb * kBlock + tok) * Hkv + g) * kTopK);
#pragma unroll
      for (int c = 0; c < 4; ++c) ids[k][c] = tok < n ? __ldg(row + c) : make_int4(-1, -1, -1, -1);
    }
    uint32_t m[kPerLane][kGroupWords];
    uint32_t left = 0;                     // bit k: token t0 + lane + 32 k not grouped yet
    bool bad = false;
#pragma unroll
    for (int k = 0; k < kPerLane; ++k) {
#pragma unroll
      for (int w = 0; w < kGroupWords; ++w) m[k][w] = 0;
      if (t0 + lane + 32 * k < n) left |= 1u << k;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int v4[4] = {ids[k][c].x, ids[k][c].y, ids[k][c].z, ids[k][c].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int b = v4[e];
          bad |= b > qb;
          const bool keep = fits && b >= 0 && b < qb;
          const uint32_t bit = keep ? (1u << (b & 31)) : 0u;
#pragma unroll
          for (int w = 0; w < kGroupWords; ++w) m[k][w] |= ((b >> 5) == w) ? bit : 0u;
        }
      }
      tok_mask[warp][lane + 32 * k] = make_uint4(m[k][0], m[k][1], m[k][2], m[k][3]);
    }
    if (bad) atomicOr(status, kStatusBounds);
    __syncwarp();
    if (!fits) {
      // ---- long sequence: consecutive tokens per tile, union built from sel
      for (int grp = 0; grp < ngrp; ++grp) {
        int* out = tile_out(grp);
        const int first = t0 + kTpt * grp;
        const int nm = min(kTpt, nw - kTpt * grp);
        const int nwords = (qb + 31) / 32;
        int cnt = 0;
        for (int w = 0; w < nwords; ++w) {
          // lane l: block 32 w + l; member i selected it?
          uint32_t tm = 0;
          for (int i = 0; i < nm; ++i) {
            const int4* row = reinterpret_cast<const int4*>(
                sel + (static_cast<size_t>(seq0 + qb * kBlock + first + i) * Hkv + g) * kTopK);
            bool hit = false;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int4 v = __ldg(row + c);
              hit |= (v.x == 32 * w + lane) | (v.y == 32 * w + lane) | (v.z == 32 * w + lane) |
                     (v.w == 32 * w + lane);
            }
            tm |= hit && (32 * w + lane < qb) ? (1u << i) : 0u;
          }
          const uint32_t bal = __ballot_sync(0xffffffffu, tm != 0u);
          if (tm) out[4 + cnt + __popc(bal & ((1u << lane) - 1u))] = ((32 * w + lane) << 8) | tm;
          cnt += __popc(bal);
        }
        if (lane == 0) {
          out[1] = 0x03020100 + 0x01010101 * first;
          out[2] = 0x07060504 + 0x01010101 * first;
          out[3] = nm;
          out[4 + cnt] = (qb << 8) | ((1 << nm) - 1);
          out[0] = cnt + 1;
        }
      }
      continue;
    }
    // ---- greedy grouping
    for (int grp = 0; grp < ngrp; ++grp) {
      const int nm = min(kTpt, nw - kTpt * grp);
      uint32_t u[kGroupWords];
      uint32_t mm[kTpt][kGroupWords];
      uint32_t offs0 = 0, offs1 = 0;
#pragma unroll
      for (int j = 0; j < kTpt; ++j) {
        int tok = 0;                       // index among the warp's tokens
        if (j < nm) {
          uint32_t key = 0xFFFFFFFFu;
          if (j == 0) {
            // seed: the lowest ungrouped token
            if (left) key = static_cast<uint32_t>(lane + 32 * (__ffs(left) - 1));
          } else {
#pragma unroll
            for (int k = 0; k < kPerLane; ++k) {
              if (left & (1u << k)) {
                int cost = 0;
#pragma unroll
                for (int w = 0; w < kGroupWords; ++w) cost += __popc(m[k][w] & ~u[w]);
                key = min(key, (static_cast<uint32_t>(cost) << 8) | static_cast<uint32_t>(lane + 32 * k));
              }
            }
          }
          tok = static_cast<int>(__reduce_min_sync(0xffffffffu, key) & 0xFFu);
          if ((tok & 31) == lane) left &= ~(1u << (tok >> 5));
          const uint4 tw = tok_mask[warp][tok];   // broadcast read
          mm[j][0] = tw.x;
          mm[j][1] = tw.y;
          mm[j][2] = tw.z;
          mm[j][3] = tw.w;
#pragma unroll
          for (int w = 0; w < kGroupWords; ++w) u[w] = (j == 0) ? mm[j][w] : (u[w] | mm[j][w]);
        } else {
#pragma unroll
          for (int w = 0; w < kGroupWords; ++w) mm[j][w] = 0;
        }
        const uint32_t off = static_cast<uint32_t>(t0 + tok);   // offset in the query block
        if (j < 4) offs0 |= off << (8 * j);
        else offs1 |= off << (8 * (j - 4));
      }
      int* out = tile_out(grp);
      if (lane == 0) {
        out[1] = static_cast<int>(offs0);
        out[2] = static_cast<int>(offs1);
        out[3] = nm;
      }
      write_union(out, mm, nm, words, qb, lane);
    }
  }
}

__global__ void __launch_bounds__(kFwdThreads, 1)
    sparse_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, const int* __restrict__ ulist,
                      int* __restrict__ tile_ctr, const int32_t* __restrict__ cu, const int2* __restrict__ tiles,
                      const int* __restrict__ num_tiles, int Hq, int Hkv, float scale,
                      __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                      uint4* __restrict__ clear, size_t clear_u16, int* __restrict__ clear_ints,
                      int n_clear_ints, uint32_t* status) {
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
      mbar_init(&sm.tile_empty[i], 2 + 8 + 1);
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
  if (clear_u16 > 0) {
    for (int i = tid; i < kZeroBytes / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(sm.zero)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();                  // the zeros -> the bulk copies' reads
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
    // to the other roles through the tile slot, -1 once none are left.  The
    // next claim's plan entry, union header and union entries (lane i: entries
    // i, i + 32, ...) are read before the current tile's K blocks are issued,
    // so those loads are in flight while K streams.
    uint32_t tcount = 0, kc = 0;
    bool alive = true;
    int pending = 0;
    if (lane == 0) pending = atomicAdd(tile_ctr + g, 1);
    pending = __shfl_sync(0xffffffffu, pending, 0);
    int2 n_pt = make_int2(0, 0);
    int n_hdr[3] = {0, 0, 0};
    int n_ent[kTpt * kTopK / 32];
    auto prefetch = [&](int ti) {
      if (ti >= total) return;
      n_pt = tiles[ti >> 4];
      const int* ul = ulist + (static_cast<size_t>(ti) * Hkv + g) * kFwdUnionStride;
      n_hdr[0] = __ldg(ul);
      n_hdr[1] = __ldg(ul + 1);
      n_hdr[2] = __ldg(ul + 2);
#pragma unroll
      for (int q = 0; q < kTpt * kTopK / 32; ++q) n_ent[q] = __ldg(ul + 4 + lane + 32 * q);
    };
    prefetch(pending);
    while (alive) {
      int ti = pending;
      TileInfo t;
      bool have = false;
      if (ti < total) {
        // the prefetched entry, if the claimed tile has tokens
        t.s = n_pt.x;
        t.qb = n_pt.y;
        t.seq0 = cu[t.s];
        t.len = cu[t.s + 1] - t.seq0;
        t.p0 = t.qb * kBlock;
        const int first = (ti & 15) * kTpt;
        t.ntok = min(kTpt, t.len - t.p0 - first);
        have = t.p0 + first < t.len;
      }
      if (!have && ti < total) {
        // a token group past the end of its query block: claim on
        if (lane == 0) {
          TileInfo tt;
          ti = atomicAdd(tile_ctr + g, 1);
          while (ti < total && !tile_info(ti, tiles, cu, tt)) ti = atomicAdd(tile_ctr + g, 1);
        }
        ti = __shfl_sync(0xffffffffu, ti, 0);
        if (ti < total) {
          tile_info(ti, tiles, cu, t);
          prefetch(ti);
        }
      }
      if (ti >= total) ti = -1;
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
      // ---- the tile's union entries (built by fwd_union_kernel)
      const int nU = min(n_hdr[0], kTpt * kTopK);
      t.offs[0] = static_cast<uint32_t>(n_hdr[1]);
      t.offs[1] = static_cast<uint32_t>(n_hdr[2]);
#pragma unroll
      for (int q = 0; q < kTpt * kTopK / 32; ++q)
        if (lane + 32 * q < nU) sm.ublk[tb][lane + 32 * q] = n_ent[q];
      if (lane == 0) {
        sm.n_union[tb] = nU;
        sm.tile_id[tb] = ti;
        sm.tinfo[tb] = t;
        pending = atomicAdd(tile_ctr + g, 1);   // next claim
      }
      pending = __shfl_sync(0xffffffffu, pending, 0);
      __syncwarp();                             // the slot is written (released by the arrive)
      if (lane == 0) mbar_arrive_expect_tx(&sm.tile_full[tb], t.ntok * 2 * kTokRows);
      __syncwarp();                             // the copies below complete after it
      // Q rows of the tile's tokens (16 heads each), one copy per token and D half
      if (lane < 2 * t.ntok) {
        const int i = lane >> 1, hf = lane & 1;
        tma_load_3d(sm.q[tb] + hf * kHalf + i * kTokRows, &tm_q, &sm.tile_full[tb], 64 * hf,
                    g * kG, t.seq0 + t.p0 + member_offset(t, i));
      }
      __syncwarp();
      prefetch(pending);                        // the next tile's entries, while K streams
      if (lane == 0) {
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
      // This CTA's share of the region to clear (the CTAs that have tiles
      // split it evenly), one 16 KB bulk copy of zeros after each V block,
      // the rest after the last one.
      const size_t ncta = static_cast<size_t>(min(static_cast<int>(gridDim.x), total)) * gridDim.y;
      const size_t cid = static_cast<size_t>(blockIdx.y) * min(static_cast<int>(gridDim.x), total) +
                         blockIdx.x;
      const size_t share = (clear_u16 + ncta - 1) / ncta;
      size_t zb = cid * share < clear_u16 ? cid * share : clear_u16;
      const size_t ze = zb + share < clear_u16 ? zb + share : clear_u16;
      // the zeros are written evict-first: they are not read before the
      // backward and should not push the forward's K and V out of L2
      const uint64_t zpol = l2_policy_evict_first();
      auto zero_one = [&]() {
        if (zb < ze) {
          const size_t n = ze - zb < kZeroBytes / 16 ? ze - zb : kZeroBytes / 16;
          bulk_store_hint(clear + zb, sm.zero, static_cast<uint32_t>(n * 16), zpol);
          bulk_commit_group();
          zb += n;
        }
      };
      if (cid == 0)
        for (int i = 0; i < n_clear_ints; ++i) clear_ints[i] = 0;
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
          zero_one();
        }
        if (!alive) break;
        mbar_arrive(&sm.tile_empty[tb]);   // done reading the tile's union list
        ++tcount;
      }
      while (zb < ze) zero_one();
      bulk_wait_all();                     // the zeros are written before the CTA exits
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
    // 1 + the Q buffer this warp's last output stores still read from (handed
    // back after the next tile's first block)
    int store_tb = 0;
    auto release_stored = [&]() {
      if (store_tb) {
        bulk_wait_read_all();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.tile_empty[store_tb - 1]);
        store_tb = 0;
      }
    };
    bool ok = true;
    for (;;) {
      const int tb = tcount & 1;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&sm.tile_full[tb], (tcount >> 1) & 1, status, 9))))
        break;
      if (sm.tile_id[tb] < 0) break;
      const TileInfo t = sm.tinfo[tb];
      const int nU = sm.n_union[tb];
      const bool row_valid = tl < t.ntok;
      const int pos = t.p0 + (row_valid ? member_offset(t, tl) : 0);
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
        if (i == 0) release_stored();
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
      // The tile's normalised O is staged in its Q buffer (free: every MMA of
      // the tile is done) in the 128B-swizzled layout of the tensor map and
      // written by one tensor store per token and half.
      uint8_t* stage = sm.q[tb] + h * kHalf;
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
          *reinterpret_cast<uint4*>(stage + sw128_offset(r, 4 * c + q)) = pk;
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();                // staged rows -> the tensor stores' reads
      mbar_arrive(&sm.o_done[h]);
      __syncwarp();
      {
        // this warp's 32 rows are tokens 2 subp and 2 subp + 1 of the tile:
        // it stores them itself, one tensor store each; the Q buffer goes back
        // to the producer once they have read it, after the next tile's first
        // block, so that the warp starts that tile without waiting for them
        const int tk = 2 * subp + lane;
        if (lane < 2 && tk < t.ntok) {
          tma_store_3d(&tm_o, stage + tk * kTokRows, 64 * h, g * kG,
                       t.seq0 + t.p0 + member_offset(t, tk));
          bulk_commit_group();
        }
        store_tb = tb + 1;
      }
      if (subp == kFirstHalfWarp % 4) {
        // one warp per half: once all the half's threads have read O, release
        // it to the next tile's PV
        bool okw = true;
        if (lane == 0) okw = mbar_wait(&sm.o_done[h], tcount & 1, status, 17);
        okw = __shfl_sync(0xffffffffu, okw ? 1 : 0, 0) != 0;
        if (okw && lane == 0) mbar_arrive(&sm.o_free);
        ok = okw;
      }
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      if (h == 0 && row_valid) lse[orow_g] = (M + __log2f(L)) * 0.6931471805599453f;
      tc_fence_before();
      ++tcount;
    }
    release_stored();
    bulk_wait_all();                           // this warp's output stores are complete
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

msa_status_t launch_sparse_fwd(const void* q, const void* k, const void* v, const int32_t* sel,
                               const int32_t* cu, int S, int T, int Hq, int Hkv, int max_seqlen,
                               float scale, const FwdWorkspace& fw, void* o, float* lse,
                               const FwdClear& clear, cudaStream_t stream) {
  if ((clear.ptr == nullptr) != (clear.bytes == 0) || clear.bytes % 16 != 0 ||
      (reinterpret_cast<uintptr_t>(clear.ptr) & 15) != 0 || clear.nints < 0 ||
      (clear.nints > 0 && clear.ints == nullptr))
    return fail(MSA_ERR_INVALID_ARG, "forward: bad region to clear");
  const Plan& plan = fw.plan;
  (void)S;
  if (Hq / Hkv != kG)
    return fail(MSA_ERR_UNSUPPORTED, "forward supports Hq/Hkv = 16 (got %d)", Hq / Hkv);
  CUtensorMap tq, tk, tv, to;
  const uint64_t dq[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hq),
                          static_cast<uint64_t>(T)};
  const uint64_t dkv[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hkv),
                           static_cast<uint64_t>(T)};
  const uint32_t bq[3] = {64, static_cast<uint32_t>(kG), 1};   // one token's 16 heads
  const uint32_t bkv[3] = {64, 1, 128};
  // o has q's layout: the same box stores one token's half rows
  if (!make_tmap_bf16(&tq, q, 3, dq, bq) || !make_tmap_bf16(&tk, k, 3, dkv, bkv) ||
      !make_tmap_bf16(&tv, v, 3, dkv, bkv) || !make_tmap_bf16(&to, o, 3, dq, bq))
    return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled failed for q/k/v/o");
  const size_t smem = sizeof(FwdSmem);
  {
    const msa_status_t e = ensure_smem(sparse_fwd_kernel, smem, "sparse_fwd_kernel");
    if (e != MSA_OK) return e;
  }
  const int per_head = (device_sm_count() + Hkv - 1) / Hkv;
  const int max_ctas = plan.max_tiles * kG;
  dim3 grid(static_cast<unsigned>(per_head < max_ctas ? per_head : max_ctas), Hkv);
  uint32_t* sw = nullptr;
  if (msa_status_t e_ = status_word(&sw); e_ != MSA_OK) return e_;
  {
    // one CTA per (128-token query block, KV head): the one-warp grouping over
    // whole blocks when sequences are long enough for its better tiles to
    // outweigh its longer serial chain (measured on 12k-token sequences)
    const int ublocks = plan.max_tiles;
    const int cap = 8 * device_sm_count();
    dim3 ugrid(static_cast<unsigned>(ublocks < cap ? ublocks : cap), Hkv);
    const bool whole = max_seqlen >= 8192;
    TraceScope trace_("fwd_union_kernel", stream);
    launch_pdl(whole ? fwd_union_kernel<1> : fwd_union_kernel<2>, ugrid, whole ? 32 : 64, 0, stream, sel, cu, plan.tiles, plan.num_tiles, Hkv,
        fw.ulist, fw.tile_ctr, sw);
  }
  {
    TraceScope trace_("sparse_fwd_kernel", stream);
    launch_pdl(sparse_fwd_kernel, grid, kFwdThreads, smem, stream,
        tq, tk, tv, to, fw.ulist, fw.tile_ctr, cu, plan.tiles, plan.num_tiles, Hq, Hkv, scale,
        static_cast<__nv_bfloat16*>(o), lse, static_cast<uint4*>(clear.ptr), clear.bytes / 16,
        clear.ints, clear.nints, sw);
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
