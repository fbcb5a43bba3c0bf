// Block-sparse GQA attention forward ("MiniMax-M3.1-Flash", 1 "Model
// Introduction": each query attends to its 16 selected 128-token blocks, own
// block included, causally; "#4581", "Kernel tuning": QSA block-sparse kernel).
//
// Tile = 128 rows = (128/G consecutive tokens) x (the G query heads of one KV
// head), so a single K/V block feeds all rows.  The tile's tokens lie in one
// 128-token block, hence share their own block.  The CTA walks the union of the
// tokens' selected blocks in ascending order; a row whose token did not select
// the current block gets P = 0 for it.  Per union block b:
//   TMA     : K_b and V_b (128 x 128 bf16 each, 128B swizzle), 2-stage ring
//   MMA     : S = Q K_b^T -> TMEM (two buffers, so S_{i+1} overlaps softmax_i)
//   softmax : thread = row = TMEM lane; running max in the log2 domain, only
//             rescaled when it grows by more than 2^8 (P stays < 256 in bf16);
//             P (bf16) written to shared memory in the MMA's K-major layout
//   MMA     : O += P V_b (V as an MN-major operand) -> TMEM
// The epilogue divides by the row sum and writes o (bf16) and lse (natural log).
#include "kernels.cuh"

namespace msa {

namespace {

constexpr int kFwdThreads = 192;            // warp 0 TMA, warp 1 MMA, warps 2..5 softmax
constexpr int kTile = 128 * 128 * 2;        // bytes of a 128 x 128 bf16 tile
constexpr int kHalf = kTile / 2;            // one 64-column half
constexpr int kMaskWords = kMaxSeqlen / kBlock / 32;
constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, false, true);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 of the largest P before a rescale

struct FwdSmem {
  uint8_t q[kTile];
  uint8_t k[2][kTile];
  uint8_t v[2][kTile];
  uint8_t p[kTile];
  uint32_t tok_mask[128][kMaskWords];       // [token of tile][block bitmap], sized for G = 1
  int ublk[kMaxSeqlen / kBlock];
  int n_union;
  uint64_t q_full;
  uint64_t kv_full[2];
  uint64_t kv_empty[2];
  uint64_t s_full[2];
  uint64_t s_empty[2];
  uint64_t p_full;
  uint64_t pv_done;
  uint32_t tmem_base;
};

}  // namespace

__global__ void __launch_bounds__(kFwdThreads, 1)
    sparse_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const int32_t* __restrict__ sel,
                      const int32_t* __restrict__ cu, const int2* __restrict__ tiles,
                      const int* __restrict__ num_tiles, int Hq, int Hkv, int G, float scale,
                      __nv_bfloat16* __restrict__ o, float* __restrict__ lse, uint32_t* status) {
  const int tpt = 128 / G;                       // tokens per tile
  const int tile_idx = blockIdx.x / G;
  const int sub = blockIdx.x % G;
  if (tile_idx >= *num_tiles) return;
  const int2 tile = tiles[tile_idx];
  const int s = tile.x, qb = tile.y, g = blockIdx.y;
  const int seq0 = cu[s];
  const int len = cu[s + 1] - seq0;
  const int p0 = qb * kBlock + sub * tpt;        // first query position of the tile
  if (p0 >= len) return;
  const int ntok = min(tpt, len - p0);
  const int nb_seq = (len + kBlock - 1) / kBlock;

  extern __shared__ uint8_t smem_raw[];
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int words = min((nb_seq + 31) >> 5, kMaskWords);

  // ---- union of the tile's selected blocks
  for (int i = tid; i < tpt * kMaskWords; i += kFwdThreads) sm.tok_mask[i / kMaskWords][i % kMaskWords] = 0;
  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.kv_full[i], 1);
      mbar_init(&sm.kv_empty[i], 1);
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_empty[i], 128);
    }
    mbar_init(&sm.p_full, 128);
    mbar_init(&sm.pv_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  for (int i = tid; i < ntok * kTopK; i += kFwdThreads) {
    const int tl = i / kTopK;
    const int b = __ldg(sel + (static_cast<size_t>(seq0 + p0 + tl) * Hkv + g) * kTopK + (i % kTopK));
    if (b < 0) continue;
    if (b > qb) {
      atomicOr(status, kStatusBounds);
      continue;
    }
    atomicOr(&sm.tok_mask[tl][b >> 5], 1u << (b & 31));
  }
  __syncthreads();
  if (warp == 0) {
    int base = 0;
    for (int w0 = 0; w0 < words; w0 += 32) {
      const int w = w0 + lane;
      uint32_t u = 0;
      if (w < words)
        for (int tl = 0; tl < ntok; ++tl) u |= sm.tok_mask[tl][w];
      const int c = __popc(u);
      int incl = c;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += n;
      }
      int off = base + incl - c;
      while (u) {
        const int bit = __ffs(u) - 1;
        sm.ublk[off++] = w * 32 + bit;
        u &= u - 1;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) sm.n_union = base;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int nU = sm.n_union;
  const uint32_t tmem = sm.tmem_base;
  const uint32_t tmem_o = tmem + 256;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (elect_one()) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(&sm.q_full, kTile);
      tma_load_3d(sm.q, &tm_q, &sm.q_full, 0, g * G, seq0 + p0);
      tma_load_3d(sm.q + kHalf, &tm_q, &sm.q_full, 64, g * G, seq0 + p0);
      for (int i = 0; i < nU; ++i) {
        const int st = i & 1;
        if (!mbar_wait(&sm.kv_empty[st], ((i >> 1) & 1) ^ 1, status)) break;
        const int row = seq0 + sm.ublk[i] * kBlock;
        mbar_arrive_expect_tx(&sm.kv_full[st], 2 * kTile);
        tma_load_3d(sm.k[st], &tm_k, &sm.kv_full[st], 0, g, row);
        tma_load_3d(sm.k[st] + kHalf, &tm_k, &sm.kv_full[st], 64, g, row);
        tma_load_3d(sm.v[st], &tm_v, &sm.kv_full[st], 0, g, row);
        tma_load_3d(sm.v[st] + kHalf, &tm_v, &sm.kv_full[st], 64, g, row);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (elect_one()) {
      bool ok = mbar_wait(&sm.q_full, 0, status);
      const uint32_t qa = smem_u32(sm.q);
      const uint32_t pa = smem_u32(sm.p);
      for (int i = 0; ok && i <= nU; ++i) {
        if (i < nU) {
          const int st = i & 1, buf = i & 1;
          ok = mbar_wait(&sm.kv_full[st], (i >> 1) & 1, status) &&
               mbar_wait(&sm.s_empty[buf], ((i >> 1) & 1) ^ 1, status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t ka = smem_u32(sm.k[st]);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            umma_bf16(tmem + buf * 128, sdesc_sw128(qa + off, 16, 1024),
                      sdesc_sw128(ka + off, 16, 1024), kIdescS, kk > 0);
          }
          umma_commit(&sm.s_full[buf]);
        }
        if (i > 0) {
          const int j = i - 1, stj = j & 1;
          ok = mbar_wait(&sm.p_full, j & 1, status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t va = smem_u32(sm.v[stj]);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t aoff = (kk >> 2) * kHalf + (kk & 3) * 32;
            umma_bf16(tmem_o, sdesc_sw128(pa + aoff, 16, 1024),
                      sdesc_sw128(va + kk * 2048, kHalf, 1024), kIdescPV, (j > 0 || kk > 0));
          }
          umma_commit(&sm.pv_done);
          umma_commit(&sm.kv_empty[stj]);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int subp = warp & 3;
    const int r = subp * 32 + lane;              // tile row = TMEM lane
    const int tl = r / G, hd = r % G;
    const bool row_valid = tl < ntok;
    const int pos = p0 + tl;
    const float sl2 = scale * kLog2e;
    const uint32_t trow = static_cast<uint32_t>(subp * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < nU; ++i) {
      const int buf = i & 1;
      const int b = sm.ublk[i];
      if (!mbar_wait(&sm.s_full[buf], (i >> 1) & 1, status)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
      float sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + trow + buf * 128 + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[c * 32 + j] = __uint_as_float(v[j]);
      }
      tc_fence_before();
      mbar_arrive(&sm.s_empty[buf]);

      const bool selected = row_valid && ((sm.tok_mask[tl][b >> 5] >> (b & 31)) & 1u);
      const int kmax = (b == qb) ? (pos & (kBlock - 1)) : (kBlock - 1);
      bool rescale = false;
      float m_use = m, rowsum = 0.f;
      if (selected) {
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 128; ++j)
          if (j <= kmax) mx = fmaxf(mx, sv[j]);
        const float m_new = fmaxf(m, mx * sl2);
        rescale = m_new > m + kRescaleThreshold;
        m_use = rescale ? m_new : m;
#pragma unroll
        for (int j = 0; j < 128; ++j) {
          const float pj = (j <= kmax) ? exp2f(fmaf(sv[j], sl2, -m_use)) : 0.f;
          sv[j] = pj;
          rowsum += pj;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 128; ++j) sv[j] = 0.f;
      }
      // O and the P buffer are free once PV of the previous block is done.
      if (i > 0) {
        if (!mbar_wait(&sm.pv_done, (i - 1) & 1, status)) { ok = false; break; }
        __syncwarp();
        tc_fence_after();
        const bool mine = rescale && m != -INFINITY;
        if (__any_sync(0xffffffffu, mine)) {
          const float alpha = mine ? exp2f(m - m_use) : 1.f;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem_o + trow + c * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
            tmem_st16(tmem_o + trow + c * 32, v);
            tmem_st16(tmem_o + trow + c * 32 + 16, v + 16);
          }
          tmem_st_wait();
        }
      }
      if (selected) {
        l = (m == -INFINITY) ? rowsum : (rescale ? l * exp2f(m - m_use) : l) + rowsum;
        m = m_use;
      }
      // P row -> shared memory (bf16, 128B-swizzled K-major, two 64-key halves)
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint4 pk;
        pk.x = pack_bf16x2(sv[8 * c + 0], sv[8 * c + 1]);
        pk.y = pack_bf16x2(sv[8 * c + 2], sv[8 * c + 3]);
        pk.z = pack_bf16x2(sv[8 * c + 4], sv[8 * c + 5]);
        pk.w = pack_bf16x2(sv[8 * c + 6], sv[8 * c + 7]);
        *reinterpret_cast<uint4*>(sm.p + (c >> 3) * kHalf + sw128_offset(r, c & 7)) = pk;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.p_full);
    }
    if (ok && mbar_wait(&sm.pv_done, (nU - 1) & 1, status)) {
      __syncwarp();
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      const size_t orow = static_cast<size_t>(seq0 + pos) * Hq + g * G + hd;
      uint4* dst = reinterpret_cast<uint4*>(o + orow * kD);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem_o + trow + c * 32, v);
        tmem_ld_wait();
        if (row_valid) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]) * inv, __uint_as_float(v[8 * j + 1]) * inv);
            pk.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]) * inv, __uint_as_float(v[8 * j + 3]) * inv);
            pk.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]) * inv, __uint_as_float(v[8 * j + 5]) * inv);
            pk.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]) * inv, __uint_as_float(v[8 * j + 7]) * inv);
            dst[c * 4 + j] = pk;
          }
        }
      }
      if (row_valid) lse[orow] = (m + __log2f(l)) * 0.6931471805599453f;
    }
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

msa_status_t launch_sparse_fwd(const void* q, const void* k, const void* v, const int32_t* sel,
                               const int32_t* cu, int S, int T, int Hq, int Hkv, int max_seqlen,
                               float scale, const Plan& plan, void* o, float* lse,
                               cudaStream_t stream) {
  (void)S;
  (void)max_seqlen;
  const int G = Hq / Hkv;
  CUtensorMap tq, tk, tv;
  const uint64_t dq[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hq),
                          static_cast<uint64_t>(T)};
  const uint64_t dkv[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hkv),
                           static_cast<uint64_t>(T)};
  const uint32_t bq[3] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(128 / G)};
  const uint32_t bkv[3] = {64, 1, 128};
  if (!make_tmap_bf16(&tq, q, 3, dq, bq) || !make_tmap_bf16(&tk, k, 3, dkv, bkv) ||
      !make_tmap_bf16(&tv, v, 3, dkv, bkv))
    return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled failed for q/k/v");
  const size_t smem = sizeof(FwdSmem) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(sparse_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    attr_set = true;
  }
  dim3 grid(plan.max_tiles * G, Hkv);
  {
    TraceScope trace_("sparse_fwd_kernel", stream);
    sparse_fwd_kernel<<<grid, kFwdThreads, smem, stream>>>(
      tq, tk, tv, sel, cu, plan.tiles, plan.num_tiles, Hq, Hkv, G, scale,
      static_cast<__nv_bfloat16*>(o), lse, status_word());
  }
  return check_launch("sparse_fwd_kernel");
}

}  // namespace msa
