// Decode step against a paged KV cache: the selection rule of "MiniMax-M3.1-Flash"
// (1 "Model Introduction": score every causal 128-token block by its max logit,
// keep the own block and the best others up to 16) applied to one new token per
// sequence, followed by its sparse attention.
//
//   decode_score_kernel  : streams the index-key cache (the bulk of the bytes,
//                          HBM-bound), one max-logit score per (seq, head, page)
//   decode_select_kernel : per (seq, KV head): the own block + the best 15
//                          earlier blocks by score (rank of each score)
//   decode_attend_kernel : per (seq, KV head, split): attention of the 16 query
//                          heads over 4 of the selected blocks with mma.sync
//                          m16n8k16 (M = 16 heads is below tcgen05's smallest M);
//                          K and V of a block arrive by TMA (128B-swizzled) into
//                          single buffers that refill while the other is in use
//   decode_merge_kernel  : combines the 4 splits' (max, sum, o)
#include "kernels.cuh"

namespace msa {

namespace {

constexpr int kPagesPerCta = 8;
constexpr int kRowPad = 136;                 // padded bf16 row (272 B) in shared memory
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ int clamp_len(int L, int max_pages, uint32_t* status) {
  if (L < 1 || L > max_pages * kBlock) {
    atomicOr(status, kStatusBounds);
    return L < 1 ? 1 : max_pages * kBlock;
  }
  return L;
}

}  // namespace

// ---------------------------------------------------------------- scores

// grid (ceil(max_pages / 8), B), 256 threads.  Warp w takes units (page, head);
// a unit is a contiguous 32 KB slab [128 keys][128 dims]; 16 lanes per key row.
__global__ void __launch_bounds__(256) decode_score_kernel(
    const __nv_bfloat16* __restrict__ q_idx, const __nv_bfloat16* __restrict__ kidx_cache,
    const int32_t* __restrict__ block_table, const int32_t* __restrict__ cache_lens, int Hkv,
    int num_pages, int max_pages, float* __restrict__ scores, uint32_t* status) {
  pdl_enter();
  const int b = blockIdx.y;
  const int L = clamp_len(cache_lens[b], max_pages, status);
  const int npages = (L + kBlock - 1) / kBlock;
  const int c0 = blockIdx.x * kPagesPerCta;
  if (c0 >= npages) return;
  const int c1 = min(npages, c0 + kPagesPerCta);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, chunk = lane & 15;
  const int units = (c1 - c0) * Hkv;
  for (int u = warp; u < units; u += 8) {
    const int c = c0 + u / Hkv, h = u % Hkv;
    int pg = block_table[static_cast<size_t>(b) * max_pages + c];
    if (pg < 0 || pg >= num_pages) {
      atomicOr(status, kStatusBounds);
      if (lane == 0) scores[(static_cast<size_t>(b) * Hkv + h) * max_pages + c] = -INFINITY;
      continue;
    }
    float qf[8];
    {
      const uint4 qv = __ldg(reinterpret_cast<const uint4*>(q_idx + (static_cast<size_t>(b) * Hkv + h) * kD) + chunk);
      const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qv);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(q2[j]);
        qf[2 * j] = f.x;
        qf[2 * j + 1] = f.y;
      }
    }
    const int nvalid = min(kBlock, L - c * kBlock);
    const uint4* slab = reinterpret_cast<const uint4*>(
        kidx_cache + (static_cast<size_t>(pg) * Hkv + h) * kBlock * kD);
    float mx = -INFINITY;
#pragma unroll 1
    for (int r0 = 0; r0 < kBlock; r0 += 16) {
      uint4 kv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) kv[i] = __ldcs(slab + (r0 + 2 * i + half) * 16 + chunk);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kv[i]);
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(k2[j]);
          acc = fmaf(qf[2 * j], f.x, fmaf(qf[2 * j + 1], f.y, acc));
        }
#pragma unroll
        for (int m = 8; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if (r0 + 2 * i + half < nvalid) mx = fmaxf(mx, acc);
      }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    if (lane == 0) scores[(static_cast<size_t>(b) * Hkv + h) * max_pages + c] = mx;
  }
}

// ---------------------------------------------------------------- select

// grid (B * Hkv), 128 threads: the own block plus the best min(15, own)
// earlier blocks by score (descending, ties: lower id); blocks b < n_init (the
// init rule, "#4581" Kernel tuning, read as: the first blocks are always kept)
// score +inf and so rank first.  Block i is kept when
// fewer than 15 blocks rank before it (higher score, or equal score and lower
// id); each thread counts for its blocks over the whole row, four scores per
// shared-memory load and four independent counters.  The kept ids are written
// ascending with the own block, -1 padded, to sel and, if given, sel_out.
__global__ void __launch_bounds__(128) decode_select_kernel(
    const float* __restrict__ scores, const int32_t* __restrict__ cache_lens, int Hkv,
    int max_pages, int n_init, int32_t* __restrict__ sel, int32_t* __restrict__ sel_out,
    uint32_t* status) {
  pdl_enter();
  __shared__ __align__(16) float key[1024];
  __shared__ int kept[16];
  __shared__ int nkept;
  const int bh = blockIdx.x;
  const int b = bh / Hkv;
  const int tid = threadIdx.x;
  const int L = clamp_len(cache_lens[b], max_pages, status);
  const int own = (L + kBlock - 1) / kBlock - 1;
  const int own4 = (own + 3) & ~3;
  const float* sc = scores + static_cast<size_t>(bh) * max_pages;
  for (int i = tid; i < own4; i += blockDim.x)
    key[i] = (i < own) ? ((i < n_init) ? INFINITY : sc[i]) : -INFINITY;
  if (tid == 0) nkept = 0;
  __syncthreads();
  for (int i = tid; i < own; i += blockDim.x) {
    const float ki = key[i];
    int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
    // padding entries (-inf at j >= own) never rank before a real block: their
    // score is not above ki and their index is not below i
#pragma unroll 4
    for (int j = 0; j < own4; j += 4) {
      const float4 k4 = *reinterpret_cast<const float4*>(&key[j]);
      c0 += (k4.x > ki || (k4.x == ki && j < i)) ? 1 : 0;
      c1 += (k4.y > ki || (k4.y == ki && j + 1 < i)) ? 1 : 0;
      c2 += (k4.z > ki || (k4.z == ki && j + 2 < i)) ? 1 : 0;
      c3 += (k4.w > ki || (k4.w == ki && j + 3 < i)) ? 1 : 0;
    }
    if (c0 + c1 + c2 + c3 < 15) kept[atomicAdd(&nkept, 1)] = i;   // at most 15 blocks
  }
  __syncthreads();
  if (tid == 0) {
    const int n = nkept;
    int v[16];
    for (int i = 0; i < 16; ++i) v[i] = (i < n) ? kept[i] : (i == n ? own : -1);
    // ascending order, -1 last (insertion sort on 16 values)
    for (int i = 1; i < 16; ++i) {
      int x = v[i], j = i - 1;
      while (j >= 0 && static_cast<unsigned>(v[j]) > static_cast<unsigned>(x)) {
        v[j + 1] = v[j];
        --j;
      }
      v[j + 1] = x;
    }
    for (int i = 0; i < 16; ++i) {
      sel[static_cast<size_t>(bh) * kTopK + i] = v[i];
      if (sel_out) sel_out[static_cast<size_t>(bh) * kTopK + i] = v[i];
    }
  }
}

// ---------------------------------------------------------------- attend

// One selected block's K or V slab (128 keys x 128 dims) as two 128B-swizzled
// 64-dim halves of 16 KB, as TMA writes them: key r, 16-byte chunk c of a half
// sits at r * 128 + ((c ^ (r % 8)) << 4).
struct AttendSmem {
  uint8_t k[2 * 16384];
  uint8_t v[2 * 16384];
  __nv_bfloat16 q[16][kRowPad];
  int page[kSplitBlocks];
  int blk[kSplitBlocks];
  uint64_t k_full, v_full;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldmatrix_x4_trans_u32(uint32_t* r, uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}

// grid (B, Hkv, kDecodeSplits), 128 threads (4 warps x 32 keys of each block):
// attention of the KV group's 16 query heads over 4 of the selected blocks.
// K and V of a block arrive by TMA into single buffers with their own
// barriers: K(i + 1) is fetched once every warp has used K(i) for S, V(i + 1)
// once P V(i) is done, so each load overlaps the other half of the block.
__global__ void __launch_bounds__(128) decode_attend_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ block_table,
    const int32_t* __restrict__ cache_lens, const int32_t* __restrict__ sel, int Hq, int Hkv,
    int num_pages, int max_pages, float scale, float* __restrict__ part_o,
    float* __restrict__ part_ml, uint32_t* status) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  AttendSmem& sm = *reinterpret_cast<AttendSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                  ~static_cast<uintptr_t>(1023));
  const int b = blockIdx.x, h = blockIdx.y, split = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = clamp_len(cache_lens[b], max_pages, status);
  const int own = (L + kBlock - 1) / kBlock - 1;
  const size_t obase = ((static_cast<size_t>(b) * Hkv + h) * kDecodeSplits + split) * 16;

  // ---- this split's blocks (sel is ascending, -1 last)
  int nmy = 0;
#pragma unroll
  for (int i = 0; i < kSplitBlocks; ++i)
    if (sel[(static_cast<size_t>(b) * Hkv + h) * kTopK + split * kSplitBlocks + i] >= 0)
      nmy = i + 1;
  if (nmy == 0) {
    for (int i = tid; i < 16; i += blockDim.x) {
      part_ml[(obase + i) * 2] = -INFINITY;
      part_ml[(obase + i) * 2 + 1] = 0.f;
    }
    return;
  }
  if (tid < kSplitBlocks) {
    const int blk =
        (tid < nmy) ? sel[(static_cast<size_t>(b) * Hkv + h) * kTopK + split * kSplitBlocks + tid] : 0;
    int pg = (tid < nmy) ? block_table[static_cast<size_t>(b) * max_pages + blk] : 0;
    if (pg < 0 || pg >= num_pages) {
      atomicOr(status, kStatusBounds);
      pg = 0;
    }
    sm.page[tid] = pg;
    sm.blk[tid] = blk;
  }
  if (tid == 0) {
    mbar_init(&sm.k_full, 1);
    mbar_init(&sm.v_full, 1);
    fence_mbar_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  __syncthreads();
  auto load = [&](const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int i) {
    const int row = (sm.page[i] * Hkv + h) * kBlock;
    mbar_arrive_expect_tx(bar, 2 * 16384);
    tma_load_2d(dst, map, bar, 0, row);
    tma_load_2d(dst + 16384, map, bar, 64, row);
  };
  if (tid == 0) {
    load(&tm_k, sm.k, &sm.k_full, 0);
    load(&tm_v, sm.v, &sm.v_full, 0);
  }
  // Q (16 heads x 128) -> padded shared rows
  for (int i = tid; i < 16 * 16; i += blockDim.x) {
    const int r = i >> 4, c = i & 15;
    *reinterpret_cast<uint4*>(&sm.q[r][c * 8]) =
        __ldg(reinterpret_cast<const uint4*>(q + (static_cast<size_t>(b) * Hq + h * 16 + r) * kD) + c);
  }
  __syncthreads();

  const int g = lane >> 2, cq = lane & 3;
  const float sl2 = scale * kLog2e;
  const uint32_t ka = smem_u32(sm.k), va = smem_u32(sm.v);
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  bool ok = true;

  for (int i = 0; i < nmy; ++i) {
    ok = mbar_wait(&sm.k_full, i & 1, status, 70);
    if (!__syncthreads_and(ok)) break;
    // S = Q K^T for this warp's 32 keys
    float s[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a[4];
      a[0] = *reinterpret_cast<const uint32_t*>(&sm.q[g][kk * 16 + 2 * cq]);
      a[1] = *reinterpret_cast<const uint32_t*>(&sm.q[g + 8][kk * 16 + 2 * cq]);
      a[2] = *reinterpret_cast<const uint32_t*>(&sm.q[g][kk * 16 + 2 * cq + 8]);
      a[3] = *reinterpret_cast<const uint32_t*>(&sm.q[g + 8][kk * 16 + 2 * cq + 8]);
      const uint8_t* kh = sm.k + (kk >> 2) * 16384;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int key = warp * 32 + nt * 8 + g;
        const int c0 = (kk & 3) * 2;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kh + swz(key, c0) + 4 * cq);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kh + swz(key, c0 + 1) + 4 * cq);
        mma_bf16_16816(s[nt], a, b0, b1);
      }
    }
    __syncthreads();                            // every warp is done with K(i)
    if (tid == 0 && i + 1 < nmy) {
      fence_proxy_async_smem();
      load(&tm_k, sm.k, &sm.k_full, i + 1);
    }
    // mask keys past the new token (own block only) and update this warp's softmax
    const int nvalid = (sm.blk[i] == own) ? (L - own * kBlock) : kBlock;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = warp * 32 + nt * 8 + 2 * cq + e;
        const bool valid = key < nvalid;
        s[nt][e] = valid ? s[nt][e] * sl2 : -INFINITY;
        s[nt][2 + e] = valid ? s[nt][2 + e] * sl2 : -INFINITY;
        mx0 = fmaxf(mx0, s[nt][e]);
        mx1 = fmaxf(mx1, s[nt][2 + e]);
      }
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, m));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, m));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float a0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0);
    const float a1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    l0 *= a0;
    l1 *= a1;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      acc[nt][0] *= a0;
      acc[nt][1] *= a0;
      acc[nt][2] *= a1;
      acc[nt][3] *= a1;
    }
    uint32_t pa[2][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p00 = (m0 == -INFINITY) ? 0.f : exp2f(s[nt][0] - m0);
      const float p01 = (m0 == -INFINITY) ? 0.f : exp2f(s[nt][1] - m0);
      const float p10 = (m1 == -INFINITY) ? 0.f : exp2f(s[nt][2] - m1);
      const float p11 = (m1 == -INFINITY) ? 0.f : exp2f(s[nt][3] - m1);
      l0 += p00 + p01;
      l1 += p10 + p11;
      // C layout of n-tiles (2kk, 2kk+1) == A layout of k-step kk
      const int kk = nt >> 1, hi = nt & 1;
      pa[kk][hi * 2 + 0] = pack_bf16x2(p00, p01);
      pa[kk][hi * 2 + 1] = pack_bf16x2(p10, p11);
    }
    ok = mbar_wait(&sm.v_full, i & 1, status, 71);
    if (!__syncthreads_and(ok)) break;
    // O += P V over this warp's 32 keys (V rows read transposed by ldmatrix)
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t a[4] = {pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3]};
      const int krow = warp * 32 + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int nt = 0; nt < 16; nt += 2) {
        const int d = nt * 8 + (lane >> 4) * 8;
        uint32_t bb[4];
        ldmatrix_x4_trans_u32(bb, va + (d >> 6) * 16384 + swz(krow, (d & 63) >> 3));
        mma_bf16_16816(acc[nt], a, bb[0], bb[1]);
        mma_bf16_16816(acc[nt + 1], a, bb[2], bb[3]);
      }
    }
    __syncthreads();                            // every warp is done with V(i)
    if (tid == 0 && i + 1 < nmy) {
      fence_proxy_async_smem();
      load(&tm_v, sm.v, &sm.v_full, i + 1);
    }
  }
  if (!ok) return;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // ---- merge the 4 warps (the K/V buffers are free: every load has landed)
  float* wo = reinterpret_cast<float*>(sm.k);     // [4][16][128]
  float* wml = wo + 4 * 16 * 128;                 // [4][16][2]
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    wo[(warp * 16 + g) * 128 + nt * 8 + 2 * cq] = acc[nt][0];
    wo[(warp * 16 + g) * 128 + nt * 8 + 2 * cq + 1] = acc[nt][1];
    wo[(warp * 16 + g + 8) * 128 + nt * 8 + 2 * cq] = acc[nt][2];
    wo[(warp * 16 + g + 8) * 128 + nt * 8 + 2 * cq + 1] = acc[nt][3];
  }
  if (cq == 0) {
    wml[(warp * 16 + g) * 2] = m0;
    wml[(warp * 16 + g) * 2 + 1] = l0;
    wml[(warp * 16 + g + 8) * 2] = m1;
    wml[(warp * 16 + g + 8) * 2 + 1] = l1;
  }
  __syncthreads();
  {
    const int hd = tid >> 3, d0 = (tid & 7) * 16;
    float mw[4], mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      mw[w] = wml[(w * 16 + hd) * 2];
      mm = fmaxf(mm, mw[w]);
    }
    float lsum = 0.f, f[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      f[w] = (mw[w] == -INFINITY) ? 0.f : exp2f(mw[w] - mm);
      lsum += f[w] * wml[(w * 16 + hd) * 2 + 1];
    }
    float* dst = part_o + (obase + hd) * kD + d0;
#pragma unroll
    for (int d = 0; d < 16; ++d) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) v += f[w] * wo[(w * 16 + hd) * 128 + d0 + d];
      dst[d] = v;
    }
    if ((tid & 7) == 0) {
      part_ml[(obase + hd) * 2] = mm;
      part_ml[(obase + hd) * 2 + 1] = lsum;
    }
  }
}

// ---------------------------------------------------------------- merge

// grid (B * Hkv), 128 threads: thread = (head, 16 channels).
__global__ void __launch_bounds__(128) decode_merge_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_ml,
                                                           int Hq, int Hkv,
                                                           __nv_bfloat16* __restrict__ o) {
  pdl_enter();
  const int bh = blockIdx.x;
  const int b = bh / Hkv, h = bh % Hkv;
  const int hd = threadIdx.x >> 3, d0 = (threadIdx.x & 7) * 16;
  float m[kDecodeSplits], mm = -INFINITY;
#pragma unroll
  for (int sp = 0; sp < kDecodeSplits; ++sp) {
    m[sp] = part_ml[((static_cast<size_t>(bh) * kDecodeSplits + sp) * 16 + hd) * 2];
    mm = fmaxf(mm, m[sp]);
  }
  float f[kDecodeSplits], l = 0.f;
#pragma unroll
  for (int sp = 0; sp < kDecodeSplits; ++sp) {
    f[sp] = (m[sp] == -INFINITY) ? 0.f : exp2f(m[sp] - mm);
    l += f[sp] * part_ml[((static_cast<size_t>(bh) * kDecodeSplits + sp) * 16 + hd) * 2 + 1];
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float out[16];
#pragma unroll
  for (int d = 0; d < 16; ++d) out[d] = 0.f;
#pragma unroll
  for (int sp = 0; sp < kDecodeSplits; ++sp) {
    if (f[sp] == 0.f) continue;
    const float* src = part_o + ((static_cast<size_t>(bh) * kDecodeSplits + sp) * 16 + hd) * kD + d0;
#pragma unroll
    for (int d = 0; d < 16; ++d) out[d] += f[sp] * src[d];
  }
  uint4* dst = reinterpret_cast<uint4*>(o + (static_cast<size_t>(b) * Hq + h * 16 + hd) * kD + d0);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint4 pk;
    pk.x = pack_bf16x2(out[8 * j + 0] * inv, out[8 * j + 1] * inv);
    pk.y = pack_bf16x2(out[8 * j + 2] * inv, out[8 * j + 3] * inv);
    pk.z = pack_bf16x2(out[8 * j + 4] * inv, out[8 * j + 5] * inv);
    pk.w = pack_bf16x2(out[8 * j + 6] * inv, out[8 * j + 7] * inv);
    dst[j] = pk;
  }
}

// ---------------------------------------------------------------- host

DecodeWorkspace carve_decode_workspace(WsCursor& ws, int B, int Hq, int Hkv, int max_pages) {
  (void)Hq;
  DecodeWorkspace w;
  w.max_pages = max_pages;
  w.scores = ws.take<float>(static_cast<size_t>(B) * Hkv * max_pages);
  w.sel = ws.take<int32_t>(static_cast<size_t>(B) * Hkv * kTopK);
  w.part_o = ws.take<float>(static_cast<size_t>(B) * Hkv * kDecodeSplits * 16 * kD);
  w.part_ml = ws.take<float>(static_cast<size_t>(B) * Hkv * kDecodeSplits * 16 * 2);
  return w;
}

msa_status_t launch_decode(const void* q, const void* q_idx, const void* k_cache,
                           const void* v_cache, const void* kidx_cache,
                           const int32_t* block_table, const int32_t* cache_lens, int B, int Hq,
                           int Hkv, int num_pages, int max_pages, float scale, int n_init,
                           void* o, int32_t* sel_out, const DecodeWorkspace& ws,
                           cudaStream_t stream) {
  uint32_t* st = nullptr;
  if (msa_status_t e_ = status_word(&st); e_ != MSA_OK) return e_;
  dim3 g1((max_pages + kPagesPerCta - 1) / kPagesPerCta, B);
  {
    TraceScope trace_("decode_score_kernel", stream);
    launch_pdl(decode_score_kernel, g1, 256, 0, stream,
        static_cast<const __nv_bfloat16*>(q_idx), static_cast<const __nv_bfloat16*>(kidx_cache),
        block_table, cache_lens, Hkv, num_pages, max_pages, ws.scores, st);
  }
  msa_status_t e = check_launch("decode_score_kernel");
  if (e != MSA_OK) return e;
  {
    TraceScope trace_("decode_select_kernel", stream);
    launch_pdl(decode_select_kernel, B * Hkv, 128, 0, stream, ws.scores, cache_lens, Hkv, max_pages,
        n_init, ws.sel, sel_out, st);
  }
  e = check_launch("decode_select_kernel");
  if (e != MSA_OK) return e;
  // K and V caches as 2-D (dims, key rows) tensors; one box = 64 dims x one block
  CUtensorMap tk, tv;
  const uint64_t dims[2] = {static_cast<uint64_t>(kD),
                            static_cast<uint64_t>(num_pages) * Hkv * kBlock};
  const uint32_t box[2] = {64, static_cast<uint32_t>(kBlock)};
  if (!make_tmap_bf16(&tk, k_cache, 2, dims, box) || !make_tmap_bf16(&tv, v_cache, 2, dims, box))
    return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the paged K/V caches");
  const size_t smem = sizeof(AttendSmem) + 1024;
  {
    const msa_status_t e = ensure_smem(decode_attend_kernel, smem, "decode_attend_kernel");
    if (e != MSA_OK) return e;
  }
  dim3 g2(B, Hkv, kDecodeSplits);
  {
    TraceScope trace_("decode_attend_kernel", stream);
    launch_pdl(decode_attend_kernel, g2, 128, smem, stream,
        tk, tv, static_cast<const __nv_bfloat16*>(q), block_table, cache_lens, ws.sel, Hq, Hkv,
        num_pages, max_pages, scale, ws.part_o, ws.part_ml, st);
  }
  e = check_launch("decode_attend_kernel");
  if (e != MSA_OK) return e;
  {
    TraceScope trace_("decode_merge_kernel", stream);
    launch_pdl(decode_merge_kernel, B * Hkv, 128, 0, stream, ws.part_o, ws.part_ml, Hq, Hkv,
        static_cast<__nv_bfloat16*>(o));
  }
  return check_launch("decode_merge_kernel");
}

}  // namespace msa

// ==================================================================== no-alloc variant
//
// msa_decode_step_static: the decode step for callers that own no device
// allocator (see msa.h).  Its scratch is the fixed array below instead of a
// caller workspace; the kernels and their launch sequence are those of
// msa_decode_step.

#include <map>
#include <mutex>

namespace msa {
namespace {

constexpr int kStaticMaxRows = 256;     // B * Hkv
constexpr int kStaticMaxPages = 1024;   // pages (128-token blocks) per sequence
constexpr size_t kStaticScores = static_cast<size_t>(kStaticMaxRows) * kStaticMaxPages;
constexpr size_t kStaticSel = static_cast<size_t>(kStaticMaxRows) * kTopK;   // int32, float-sized
constexpr size_t kStaticPartO = static_cast<size_t>(kStaticMaxRows) * kDecodeSplits * 16 * kD;
constexpr size_t kStaticPartMl = static_cast<size_t>(kStaticMaxRows) * kDecodeSplits * 16 * 2;

// One copy per GPU that loads the library, kept until the process exits
// (about 9.6 MB).  In host code this name is only a host-side stand-in for
// the symbol: kernels must be given the device address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) float g_decode_scratch[kStaticScores + kStaticSel +
                                                        kStaticPartO + kStaticPartMl];

std::mutex g_static_mu;
std::map<unsigned long long, float*> g_static_ptr;   // context id -> device address

// Device address of g_decode_scratch in the calling thread's current context.
// Looked up with cudaGetSymbolAddress on the first call in each context (so
// once per device, with that device current) and cached under the context's
// process-unique id: a context made after cudaDeviceReset, whose module may
// sit at another address, gets a fresh lookup instead of the stale one.
msa_status_t static_scratch(float** out) {
  unsigned long long ctx = 0;
  msa_status_t st = current_context_id(&ctx);
  if (st != MSA_OK) return st;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (ctx != 0) {
    auto it = g_static_ptr.find(ctx);
    if (it != g_static_ptr.end()) {
      *out = it->second;
      return MSA_OK;
    }
  }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess || p == nullptr)
    return fail(MSA_ERR_CUDA, "cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(e));
  if (ctx == 0) {                 // the lookup made the device's primary context current
    st = current_context_id(&ctx);
    if (st != MSA_OK) return st;
  }
  if (ctx != 0) g_static_ptr[ctx] = static_cast<float*>(p);
  *out = static_cast<float*>(p);
  return MSA_OK;
}

}  // namespace
}  // namespace msa

extern "C" msa_status_t msa_decode_step_static(const void* q, const void* q_idx,
                                               const void* k_cache, const void* v_cache,
                                               const void* kidx_cache,
                                               const int32_t* block_table,
                                               const int32_t* cache_lens, int B, int Hq,
                                               int Hkv, int num_pages, int max_pages,
                                               float scale, void* o, int32_t* sel_out,
                                               msa_stream_t stream) {
  using namespace msa;
  const void* ptrs[] = {q, q_idx, k_cache, v_cache, kidx_cache, block_table, cache_lens, o};
  const char* names[] = {"q", "q_idx", "k_cache", "v_cache", "kidx_cache", "block_table",
                         "cache_lens", "o"};
  for (int i = 0; i < 8; ++i)
    if (!ptrs[i] || !aligned16(ptrs[i]))
      return fail(MSA_ERR_INVALID_ARG, "%s is null or not 16-byte aligned", names[i]);
  if (sel_out && !aligned16(sel_out))
    return fail(MSA_ERR_INVALID_ARG, "sel_out is not 16-byte aligned");
  if (B < 1 || num_pages < 1 || max_pages < 1)
    return fail(MSA_ERR_INVALID_ARG, "B, num_pages and max_pages must be >= 1");
  if (Hq < 1 || Hkv < 1 || Hq != 16 * Hkv)
    return fail(MSA_ERR_UNSUPPORTED, "decode needs Hq = 16 * Hkv (got Hq %d, Hkv %d)", Hq, Hkv);
  if (!(scale > 0.0f)) return fail(MSA_ERR_INVALID_ARG, "scale must be > 0");
  if (static_cast<long long>(B) * Hkv > kStaticMaxRows)
    return fail(MSA_ERR_UNSUPPORTED,
                "msa_decode_step_static holds scratch for B * Hkv <= %d (got %d x %d); "
                "use msa_decode_step with a workspace",
                kStaticMaxRows, B, Hkv);
  if (max_pages > kStaticMaxPages)
    return fail(MSA_ERR_UNSUPPORTED,
                "msa_decode_step_static holds scratch for max_pages <= %d (got %d); "
                "use msa_decode_step with a workspace",
                kStaticMaxPages, max_pages);
  float* base = nullptr;
  msa_status_t st = static_scratch(&base);
  if (st != MSA_OK) return st;
  DecodeWorkspace ws;
  ws.max_pages = max_pages;
  ws.scores = base;                                   // [B, Hkv, max_pages]
  ws.sel = reinterpret_cast<int32_t*>(base + kStaticScores);                    // [B, Hkv, 16]
  ws.part_o = base + kStaticScores + kStaticSel;                                // [B, Hkv, splits, 16, 128]
  ws.part_ml = base + kStaticScores + kStaticSel + kStaticPartO;                // [B, Hkv, splits, 16, 2]
  return launch_decode(q, q_idx, k_cache, v_cache, kidx_cache, block_table, cache_lens, B, Hq,
                       Hkv, num_pages, max_pages, scale, 0, o, sel_out, ws,
                       static_cast<cudaStream_t>(stream));
}
