// Decode step against a paged KV cache: the selection rule of "MiniMax-M3.1-Flash"
// (1 "Model Introduction": score every causal 128-token block by its max logit,
// keep the own block and the best others up to 16) applied to one new token per
// sequence, followed by its sparse attention.
//
//   decode_score_kernel  : streams the index-key cache (the bulk of the bytes,
//                          HBM-bound), one max-logit score per (seq, head, page)
//   decode_attend_kernel : per (seq, KV head, split): top-15 + own block from the
//                          scores (bitonic sort in shared memory), then
//                          attention of the 16 query heads over 4 of the
//                          selected pages with mma.sync m16n8k16 (M = 16 heads
//                          is below tcgen05's smallest M), per-warp online
//                          softmax, cp.async double buffering
//   decode_merge_kernel  : combines the 4 splits' (max, sum, o)
#include "kernels.cuh"

namespace msa {

namespace {

constexpr int kPagesPerCta = 8;
constexpr int kRowPad = 136;                 // padded bf16 row (272 B) in shared memory
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
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

// ---------------------------------------------------------------- select + attend

struct AttendSmem {
  __nv_bfloat16 q[16][kRowPad];
  __nv_bfloat16 kv[2][2][kBlock][kRowPad];     // [buffer][K or V][key][dim]
  float key[1024];
  int id[1024];
  int chosen[16];
};

__global__ void __launch_bounds__(128) decode_attend_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_cache,
    const __nv_bfloat16* __restrict__ v_cache, const int32_t* __restrict__ block_table,
    const int32_t* __restrict__ cache_lens, int Hq, int Hkv, int num_pages, int max_pages,
    float scale, const float* __restrict__ scores, int32_t* __restrict__ sel_out,
    float* __restrict__ part_o, float* __restrict__ part_ml, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  AttendSmem& sm = *reinterpret_cast<AttendSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                                  ~static_cast<uintptr_t>(127));
  const int b = blockIdx.x, h = blockIdx.y, split = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = clamp_len(cache_lens[b], max_pages, status);
  const int nb = (L + kBlock - 1) / kBlock;
  const int own = nb - 1;

  // ---- top-15 earlier blocks by score (descending, ties: lower id), then own
  int n2 = 1;
  while (n2 < own) n2 <<= 1;
  const float* sc = scores + (static_cast<size_t>(b) * Hkv + h) * max_pages;
  for (int i = tid; i < n2; i += 128) {
    sm.key[i] = (i < own) ? sc[i] : -INFINITY;
    sm.id[i] = (i < own) ? i : 0x7fffffff;
  }
  __syncthreads();
  for (int kk = 2; kk <= n2; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < n2; i += 128) {
        const int l = i ^ j;
        if (l > i) {
          const float ki = sm.key[i], kl = sm.key[l];
          const int ii = sm.id[i], il = sm.id[l];
          // "i before l" in the target order: higher score, then lower id
          const bool l_first = (kl > ki) || (kl == ki && il < ii);
          const bool desc = (i & kk) == 0;
          if (desc ? l_first : !l_first) {
            sm.key[i] = kl;
            sm.key[l] = ki;
            sm.id[i] = il;
            sm.id[l] = ii;
          }
        }
      }
      __syncthreads();
    }
  }
  if (tid == 0) {
    int v[16];
    const int nkeep = min(15, own);
    for (int i = 0; i < 16; ++i) v[i] = (i < nkeep) ? sm.id[i] : (i == nkeep ? own : -1);
    // ascending order, -1 last (insertion sort on 16 values)
    for (int i = 1; i < 16; ++i) {
      int x = v[i], j = i - 1;
      while (j >= 0 && static_cast<unsigned>(v[j]) > static_cast<unsigned>(x)) {
        v[j + 1] = v[j];
        --j;
      }
      v[j + 1] = x;
    }
    for (int i = 0; i < 16; ++i) sm.chosen[i] = v[i];
    if (split == 0 && sel_out)
      for (int i = 0; i < 16; ++i) sel_out[(static_cast<size_t>(b) * Hkv + h) * kTopK + i] = v[i];
  }
  __syncthreads();

  // ---- this split's blocks
  int my_blk[4], nmy = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int blk = sm.chosen[split * 4 + i];
    my_blk[i] = blk;
    if (blk >= 0) nmy = i + 1;
  }
  int my_page[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int pg = (i < nmy) ? block_table[static_cast<size_t>(b) * max_pages + my_blk[i]] : 0;
    if (pg < 0 || pg >= num_pages) {
      atomicOr(status, kStatusBounds);
      pg = 0;
    }
    my_page[i] = pg;
  }
  const size_t obase = ((static_cast<size_t>(b) * Hkv + h) * kDecodeSplits + split) * 16;
  if (nmy == 0) {
    for (int i = tid; i < 16; i += 128) {
      part_ml[(obase + i) * 2] = -INFINITY;
      part_ml[(obase + i) * 2 + 1] = 0.f;
    }
    return;
  }

  // Q (16 heads x 128) -> shared
  for (int i = tid; i < 16 * 16; i += 128) {
    const int r = i >> 4, c = i & 15;
    cp_async16(&sm.q[r][c * 8], q + (static_cast<size_t>(b) * Hq + h * 16 + r) * kD + c * 8);
  }
  auto load_block = [&](int i, int buf) {
    const size_t base = (static_cast<size_t>(my_page[i]) * Hkv + h) * kBlock * kD;
    for (int x = tid; x < 2 * kBlock * 16; x += 128) {
      const int which = x >> 11, rr = (x >> 4) & 127, c = x & 15;
      const __nv_bfloat16* src = (which ? v_cache : k_cache) + base + rr * kD + c * 8;
      cp_async16(&sm.kv[buf][which][rr][c * 8], src);
    }
  };
  load_block(0, 0);
  cp_async_commit();

  const int g = lane >> 2, cq = lane & 3;
  const float sl2 = scale * kLog2e;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

  for (int i = 0; i < nmy; ++i) {
    const int buf = i & 1;
    if (i + 1 < nmy) {
      load_block(i + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
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
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int key = warp * 32 + nt * 8 + g;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&sm.kv[buf][0][key][kk * 16 + 2 * cq]);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&sm.kv[buf][0][key][kk * 16 + 2 * cq + 8]);
        mma_bf16_16816(s[nt], a, b0, b1);
      }
    }
    // mask keys past the new token (own block only) and update this warp's softmax
    const int nvalid = (my_blk[i] == own) ? (L - own * kBlock) : kBlock;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = warp * 32 + nt * 8 + 2 * cq + e;
        const bool ok = key < nvalid;
        s[nt][e] = ok ? s[nt][e] * sl2 : -INFINITY;
        s[nt][2 + e] = ok ? s[nt][2 + e] * sl2 : -INFINITY;
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
    // O += P V over this warp's 32 keys
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t a[4] = {pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3]};
      const int krow = warp * 32 + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int nt = 0; nt < 16; nt += 2) {
        uint32_t bb[4];
        ldmatrix_x4_trans(bb, &sm.kv[buf][1][krow][nt * 8 + (lane >> 4) * 8]);
        mma_bf16_16816(acc[nt], a, bb[0], bb[1]);
        mma_bf16_16816(acc[nt + 1], a, bb[2], bb[3]);
      }
    }
    __syncthreads();
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // ---- merge the 4 warps (shared memory reused)
  float* wo = reinterpret_cast<float*>(&sm.kv[0][0][0][0]);     // [4][16][128]
  float* wml = wo + 4 * 16 * 128;                                // [4][16][2]
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
  w.part_o = ws.take<float>(static_cast<size_t>(B) * Hkv * kDecodeSplits * 16 * kD);
  w.part_ml = ws.take<float>(static_cast<size_t>(B) * Hkv * kDecodeSplits * 16 * 2);
  return w;
}

msa_status_t launch_decode(const void* q, const void* q_idx, const void* k_cache,
                           const void* v_cache, const void* kidx_cache,
                           const int32_t* block_table, const int32_t* cache_lens, int B, int Hq,
                           int Hkv, int num_pages, int max_pages, float scale, void* o,
                           int32_t* sel_out, const DecodeWorkspace& ws, cudaStream_t stream) {
  uint32_t* st = status_word();
  dim3 g1((max_pages + kPagesPerCta - 1) / kPagesPerCta, B);
  {
    TraceScope trace_("decode_score_kernel", stream);
    decode_score_kernel<<<g1, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(q_idx), static_cast<const __nv_bfloat16*>(kidx_cache),
      block_table, cache_lens, Hkv, num_pages, max_pages, ws.scores, st);
  }
  msa_status_t e = check_launch("decode_score_kernel");
  if (e != MSA_OK) return e;
  const size_t smem = sizeof(AttendSmem) + 128;
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(decode_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    attr_set = true;
  }
  dim3 g2(B, Hkv, kDecodeSplits);
  {
    TraceScope trace_("decode_attend_kernel", stream);
    decode_attend_kernel<<<g2, 128, smem, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_cache),
      static_cast<const __nv_bfloat16*>(v_cache), block_table, cache_lens, Hq, Hkv, num_pages,
      max_pages, scale, ws.scores, sel_out, ws.part_o, ws.part_ml, st);
  }
  e = check_launch("decode_attend_kernel");
  if (e != MSA_OK) return e;
  {
    TraceScope trace_("decode_merge_kernel", stream);
    decode_merge_kernel<<<B * Hkv, 128, 0, stream>>>(ws.part_o, ws.part_ml, Hq, Hkv,
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

#include <mutex>

namespace msa {
namespace {

constexpr int kStaticMaxRows = 256;     // B * Hkv
constexpr int kStaticMaxPages = 1024;   // pages (128-token blocks) per sequence
constexpr size_t kStaticScores = static_cast<size_t>(kStaticMaxRows) * kStaticMaxPages;
constexpr size_t kStaticPartO = static_cast<size_t>(kStaticMaxRows) * kDecodeSplits * 16 * kD;
constexpr size_t kStaticPartMl = static_cast<size_t>(kStaticMaxRows) * kDecodeSplits * 16 * 2;

// One copy per GPU that loads the library, kept until the process exits
// (about 9.2 MB).  In host code this name is only a host-side stand-in for
// the symbol: kernels must be given the device address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) float g_decode_scratch[kStaticScores + kStaticPartO +
                                                        kStaticPartMl];

std::mutex g_static_mu;
float* g_static_ptr[64] = {nullptr};

// Device address of g_decode_scratch on the current device, looked up once
// per device (with that device current) and cached.
msa_status_t static_scratch(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(MSA_ERR_UNSUPPORTED, "device index %d above 63", dev);
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(MSA_ERR_CUDA, "cudaGetSymbolAddress(decode scratch): %s",
                  cudaGetErrorString(e));
    g_static_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_static_ptr[dev];
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
  ws.part_o = base + kStaticScores;                   // [B, Hkv, splits, 16, 128]
  ws.part_ml = base + kStaticScores + kStaticPartO;   // [B, Hkv, splits, 16, 2]
  return launch_decode(q, q_idx, k_cache, v_cache, kidx_cache, block_table, cache_lens, B, Hq,
                       Hkv, num_pages, max_pages, scale, o, sel_out, ws,
                       static_cast<cudaStream_t>(stream));
}
