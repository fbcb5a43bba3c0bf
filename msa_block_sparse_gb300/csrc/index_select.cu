// Index select: for every (token, index head) score each earlier 128-token key
// block of the token's sequence by its maximum logit q_idx . k_idx and keep the
// own block plus the 15 best earlier blocks ("MiniMax-M3.1-Flash", 1 "Model
// Introduction"; "#4581", "Kernel tuning": per-block max logits then top-k).
//
// One CTA per (128-token query tile, index head).  All tokens of a tile share
// their own block qb, so every earlier block b < qb is fully causal for every
// row and the own block needs no score (it is always kept).  For b = 0..qb-1:
//   TMA    : K block b (128 x 128 bf16, 128B swizzle) into a 4-stage ring
//   MMA    : S_b = Q K_b^T (M = N = K = 128) into one of two TMEM buffers
//   epilogue (4 warps, thread = query row = TMEM lane): row max of S_b,
//            then a register-resident insertion into a descending top-15
//            list (strictly greater wins, so equal scores keep the lower id).
// With the init rule ("#4581", Kernel tuning; read as: the first n_init
// blocks are always kept) blocks b < n_init enter the list with score +inf,
// so they take the first places and the best others fill the rest.
// The scores never leave the SM.
#include "kernels.cuh"

namespace msa {

namespace {

constexpr int kSelStages = 4;
constexpr int kSelThreads = 192;         // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kTileBytes = 128 * 128 * 2;  // one 128 x 128 bf16 tile
constexpr uint32_t kSelIdesc = idesc_bf16(128, 128, false, false);

struct SelSmem {
  uint8_t q[kTileBytes];
  uint8_t k[kSelStages][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[kSelStages];
  uint64_t k_empty[kSelStages];
  uint64_t s_full[2];
  uint64_t s_empty[2];
  uint32_t tmem_base;
};

__device__ __forceinline__ void cswap(int& a, int& b) {
  // ascending, with -1 (unused) sorted to the end
  const unsigned ua = static_cast<unsigned>(a), ub = static_cast<unsigned>(b);
  if (ua > ub) {
    int t = a;
    a = b;
    b = t;
  }
}

__device__ __forceinline__ void write_selection(int32_t* out, int own, const int* ids) {
  int v[16];
  v[0] = own;
#pragma unroll
  for (int i = 0; i < 15; ++i) v[i + 1] = ids[i];
  // bitonic sort of 16 values (as unsigned: -1 sorts last)
#pragma unroll
  for (int k = 2; k <= 16; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int l = i ^ j;
        if (l > i) {
          if ((i & k) == 0) cswap(v[i], v[l]);
          else cswap(v[l], v[i]);
        }
      }
    }
  }
  int4* o4 = reinterpret_cast<int4*>(out);
#pragma unroll
  for (int i = 0; i < 4; ++i) o4[i] = make_int4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

}  // namespace

__global__ void __launch_bounds__(kSelThreads, 1)
    index_select_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, const int32_t* __restrict__ cu,
                        const int2* __restrict__ tiles, const int* __restrict__ num_tiles, int Hi,
                        int n_init, int32_t* __restrict__ sel, uint32_t* status) {
  pdl_enter();
  if (static_cast<int>(blockIdx.x) >= *num_tiles) return;
  extern __shared__ uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const int2 tile = tiles[blockIdx.x];
  const int s = tile.x, qb = tile.y, h = blockIdx.y;
  const int seq0 = cu[s];
  const int len = cu[s + 1] - seq0;
  const int row0 = qb * kBlock;                     // first query position of the tile
  const int nrows = min(kBlock, len - row0);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (qb == 0) {   // only the own block exists
    if (threadIdx.x < nrows) {
      int ids[15];
#pragma unroll
      for (int i = 0; i < 15; ++i) ids[i] = -1;
      write_selection(sel + (static_cast<size_t>(seq0 + threadIdx.x) * Hi + h) * kTopK, 0, ids);
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    for (int i = 0; i < kSelStages; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_empty[i], 128);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int nblk = qb;   // scored blocks 0 .. qb-1

  if (warp == 0) {
    if (elect_one()) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
      tma_load_3d(sm.q, &tm_q, &sm.q_full, 0, h, seq0 + row0);
      tma_load_3d(sm.q + kTileBytes / 2, &tm_q, &sm.q_full, 64, h, seq0 + row0);
      for (int b = 0; b < nblk; ++b) {
        const int st = b % kSelStages;
        if (!mbar_wait(&sm.k_empty[st], ((b / kSelStages) & 1) ^ 1, status)) break;
        mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
        tma_load_3d(sm.k[st], &tm_k, &sm.k_full[st], 0, h, seq0 + b * kBlock);
        tma_load_3d(sm.k[st] + kTileBytes / 2, &tm_k, &sm.k_full[st], 64, h, seq0 + b * kBlock);
      }
    }
  } else if (warp == 1) {
    if (elect_one()) {
      bool ok = mbar_wait(&sm.q_full, 0, status);
      const uint32_t qa = smem_u32(sm.q);
      for (int b = 0; ok && b < nblk; ++b) {
        const int st = b % kSelStages, buf = b & 1;
        ok = mbar_wait(&sm.k_full[st], (b / kSelStages) & 1, status) &&
             mbar_wait(&sm.s_empty[buf], ((b >> 1) & 1) ^ 1, status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ka = smem_u32(sm.k[st]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
          umma_bf16(tmem + buf * 128, sdesc_sw128(qa + off, 16, 1024),
                    sdesc_sw128(ka + off, 16, 1024), kSelIdesc, kk > 0);
        }
        umma_commit(&sm.k_empty[st]);
        umma_commit(&sm.s_full[buf]);
      }
    }
  } else {
    // epilogue: thread = query row = TMEM lane
    const int sub = warp & 3;                 // TMEM sub-partition of this warp
    const int r = sub * 32 + lane;
    float best[15];
    int ids[15];
#pragma unroll
    for (int i = 0; i < 15; ++i) {
      best[i] = -INFINITY;
      ids[i] = -1;
    }
    const uint32_t trow = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    for (int b = 0; b < nblk; ++b) {
      const int buf = b & 1;
      if (!mbar_wait(&sm.s_full[buf], (b >> 1) & 1, status)) break;
      __syncwarp();
      tc_fence_after();
      // all 128 columns in flight at once, one wait, then the buffer is free
      // for the MMA two blocks ahead while the row max is taken
      uint32_t v[128];
#pragma unroll
      for (int c = 0; c < 128; c += 32) tmem_ld32(trow + buf * 128 + c, v + c);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&sm.s_empty[buf]);
      float m4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t* w = v + 32 * q;
        float t = max3f(__uint_as_float(w[0]), __uint_as_float(w[1]), __uint_as_float(w[2]));
#pragma unroll
        for (int j = 3; j < 31; j += 2)
          t = max3f(t, __uint_as_float(w[j]), __uint_as_float(w[j + 1]));
        m4[q] = fmaxf(t, __uint_as_float(w[31]));
      }
      const float mx = (b < n_init) ? INFINITY : fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      float cv = mx;
      int ci = b;
#pragma unroll
      for (int i = 0; i < 15; ++i) {
        if (cv > best[i]) {
          const float tv = best[i];
          const int ti = ids[i];
          best[i] = cv;
          ids[i] = ci;
          cv = tv;
          ci = ti;
        }
      }
    }
    if (r < nrows)
      write_selection(sel + (static_cast<size_t>(seq0 + row0 + r) * Hi + h) * kTopK, qb, ids);
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

msa_status_t launch_index_select(const void* q_idx, const void* k_idx, const int32_t* cu, int S,
                                 int T, int Hi, int n_init, const Plan& plan, int32_t* sel,
                                 cudaStream_t stream) {
  (void)S;
  CUtensorMap tq, tk;
  const uint64_t dims[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hi),
                            static_cast<uint64_t>(T)};
  const uint32_t box[3] = {64, 1, 128};
  if (!make_tmap_bf16(&tq, q_idx, 3, dims, box) || !make_tmap_bf16(&tk, k_idx, 3, dims, box))
    return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled failed for q_idx/k_idx");
  const size_t smem = sizeof(SelSmem) + 1024;
  {
    const msa_status_t e = ensure_smem(index_select_kernel, smem, "index_select_kernel");
    if (e != MSA_OK) return e;
  }
  uint32_t* sw = nullptr;
  if (msa_status_t e_ = status_word(&sw); e_ != MSA_OK) return e_;
  dim3 grid(plan.max_tiles, Hi);
  {
    TraceScope trace_("index_select_kernel", stream);
    launch_pdl(index_select_kernel, grid, kSelThreads, smem, stream, tq, tk, cu, plan.tiles,
        plan.num_tiles, Hi, n_init, sel, sw);
  }
  return check_launch("index_select_kernel");
}

}  // namespace msa
