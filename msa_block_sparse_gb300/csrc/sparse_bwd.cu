// Block-sparse attention backward ("#4581", "Kernel tuning": dQ and dK/dV of
// the block-sparse kernel; "MiniMax-M3.1-Flash", 5.4 "Notable quirks": the
// indexer is frozen, so the selection is a constant here).
//
// KV-major schedule.  A work item is (KV head g, key block b of sequence s, a
// segment of candidate query positions).  Its CTA keeps K_b and V_b in shared
// memory and streams the query tokens of the segment that selected b, in
// ascending order, in chunks of 128/G tokens x G heads = 128 columns:
//   scanner  : warp 0 reads each candidate's 16 selected ids, compacts the
//              matches with a ballot, loads the chunk's Q and dO rows by TMA
//              and its lse / Delta values into shared memory
//   MMA      : S^T = K_b Q^T and dP^T = V_b dO^T (M = keys, N = columns)
//   compute  : thread = key; P^T = exp2(S^T log2e scale - lse log2e) masked
//              causally, dS^T = P^T (dP^T - Delta); both as bf16 in shared
//              memory (one buffer serves as K-major and MN-major operand)
//   MMA      : dV += P^T dO, dK += dS^T Q (TMEM accumulators over the whole
//              item), dQ^T = K_b^T dS^T (M = head dim, N = columns)
//   compute  : dQ^T drained from TMEM into the fp32 dQ accumulator with
//              coalesced atomics (a warp covers 32 consecutive channels)
// At the end of the item dK and dV are added to fp32 accumulators (segments
// of one block add up there); a last kernel scales and converts to bf16.
#include "kernels.cuh"

namespace msa {

namespace {

constexpr int kBwdThreads = 192;            // warp 0 scan + TMA, warp 1 MMA, warps 2..5 compute
constexpr int kTile = 128 * 128 * 2;
constexpr int kHalf = kTile / 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kIdescKK = idesc_bf16(128, 128, false, false);   // both K-major
constexpr uint32_t kIdescKM = idesc_bf16(128, 128, false, true);    // B MN-major
constexpr uint32_t kIdescMM = idesc_bf16(128, 128, true, true);     // both MN-major

struct BwdSmem {
  uint8_t k[kTile];
  uint8_t v[kTile];
  uint8_t q[kTile];
  uint8_t dout[kTile];
  uint8_t pt[kTile];
  uint8_t dst[kTile];
  float lse2[128];
  float delta[128];
  int tok[16];
  int ntok;
  uint64_t kv_full;
  uint64_t ld_full;
  uint64_t ld_empty;
  uint64_t st_full;
  uint64_t ds_full;
  uint64_t mm_done;
  uint64_t dq_free;
  uint32_t tmem_base;
};

}  // namespace

// ---------------------------------------------------------------- items

// One CTA: turns the tile plan (qb descending) into work items with the key
// block ascending, each block split into segments of kBwdSegment candidate
// query positions [128 b, len).
__global__ void __launch_bounds__(1024) bwd_items_kernel(const int32_t* __restrict__ cu,
                                                         const int2* __restrict__ tiles,
                                                         const int* __restrict__ num_tiles,
                                                         int4* __restrict__ items,
                                                         int* __restrict__ num_items,
                                                         int max_items, uint32_t* status) {
  __shared__ int warp_sums[32];
  __shared__ int carry;
  const int n = *num_tiles;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < n; base += blockDim.x) {
    const int j = base + threadIdx.x;
    int s = 0, b = 0, len = 0, nseg = 0;
    if (j < n) {
      const int2 t = tiles[n - 1 - j];
      s = t.x;
      b = t.y;
      len = cu[s + 1] - cu[s];
      nseg = (len - b * kBlock + kBwdSegment - 1) / kBwdSegment;
    }
    // block-wide exclusive scan of nseg
    int incl = nseg;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += x;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
      int ws = (lane < static_cast<int>(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, ws, d);
        if (lane >= d) ws += x;
      }
      warp_sums[lane] = ws;
    }
    __syncthreads();
    const int off = carry + (w > 0 ? warp_sums[w - 1] : 0) + incl - nseg;
    for (int k = 0; k < nseg; ++k) {
      const int idx = off + k;
      const int p0 = b * kBlock + k * kBwdSegment;
      if (idx < max_items) items[idx] = make_int4(s, b, p0, min(len, p0 + kBwdSegment));
      else atomicOr(status, kStatusBounds);
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = off + nseg;
    __syncthreads();
  }
  if (threadIdx.x == 0) *num_items = min(carry, max_items);
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
                      const __grid_constant__ CUtensorMap tm_do, const int32_t* __restrict__ sel,
                      const int32_t* __restrict__ cu, const float* __restrict__ lse,
                      const float* __restrict__ delta, const int4* __restrict__ items,
                      const int* __restrict__ num_items, int Hq, int Hkv, int G, float scale,
                      float* __restrict__ dq_acc, float* __restrict__ dk_acc,
                      float* __restrict__ dv_acc, uint32_t* status) {
  if (static_cast<int>(blockIdx.x) >= *num_items) return;
  const int4 item = items[blockIdx.x];
  const int s = item.x, b = item.y, pbeg = item.z, pend = item.w;
  const int g = blockIdx.y;
  const int seq0 = cu[s];
  const int len = cu[s + 1] - seq0;
  const int tpt = 128 / G;

  extern __shared__ uint8_t smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.ld_full, 1);
    mbar_init(&sm.ld_empty, 1);
    mbar_init(&sm.st_full, 1);
    mbar_init(&sm.ds_full, 128);
    mbar_init(&sm.mm_done, 1);
    mbar_init(&sm.dq_free, 128);
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
  const uint32_t t_dv = tmem, t_dk = tmem + 128, t_s = tmem + 256, t_dp = tmem + 384;

  if (warp == 0) {
    // ------------------------------------------------------------ scanner / TMA
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_do);
      mbar_arrive_expect_tx(&sm.kv_full, 2 * kTile);
      const int row = seq0 + b * kBlock;
      tma_load_3d(sm.k, &tm_k, &sm.kv_full, 0, g, row);
      tma_load_3d(sm.k + kHalf, &tm_k, &sm.kv_full, 64, g, row);
      tma_load_3d(sm.v, &tm_v, &sm.kv_full, 0, g, row);
      tma_load_3d(sm.v + kHalf, &tm_v, &sm.kv_full, 64, g, row);
    }
    int chunk = 0, cnt = 0, my_pos = -1;
    bool alive = true;
    auto emit = [&](int n) {
      // wait until the previous chunk's MMAs have released the Q/dO buffer
      if (lane == 0) alive = mbar_wait(&sm.ld_empty, (chunk & 1) ^ 1, status);
      alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
      if (!alive) return;
      const int first = __shfl_sync(0xffffffffu, my_pos, 0);
      const int pos = (lane < n) ? my_pos : first;
      if (lane < tpt) {
        sm.tok[lane] = (lane < n) ? pos : -1;
        const size_t base = static_cast<size_t>(seq0 + pos) * Hq + g * G;
        for (int h = 0; h < G; ++h) {
          sm.lse2[lane * G + h] = __ldg(lse + base + h) * kLog2e;
          sm.delta[lane * G + h] = __ldg(delta + base + h);
        }
      }
      if (lane == 0) sm.ntok = n;
      __syncwarp();
      if (n > 0) {
        int slot_pos[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) slot_pos[i] = __shfl_sync(0xffffffffu, pos, i);
        if (lane == 0) {
          mbar_arrive_expect_tx(&sm.ld_full, 2 * kTile);
          for (int i = 0; i < tpt; ++i) {
            const int t = seq0 + slot_pos[i];
            const uint32_t off = i * G * 128;
            tma_load_3d(sm.q + off, &tm_q, &sm.ld_full, 0, g * G, t);
            tma_load_3d(sm.q + kHalf + off, &tm_q, &sm.ld_full, 64, g * G, t);
            tma_load_3d(sm.dout + off, &tm_do, &sm.ld_full, 0, g * G, t);
            tma_load_3d(sm.dout + kHalf + off, &tm_do, &sm.ld_full, 64, g * G, t);
          }
        }
      } else if (lane == 0) {
        mbar_arrive(&sm.ld_full);   // end marker: no data
      }
      ++chunk;
    };
    for (int base = pbeg; alive && base < pend; base += 32) {
      const int p = base + lane;
      bool hit = false;
      if (p < pend) {
        const int4* row = reinterpret_cast<const int4*>(
            sel + (static_cast<size_t>(seq0 + p) * Hkv + g) * kTopK);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int4 v = __ldg(row + c);
          hit |= (v.x == b) | (v.y == b) | (v.z == b) | (v.w == b);
        }
      }
      uint32_t mask = __ballot_sync(0xffffffffu, hit);
      while (mask) {
        const int bit = __ffs(mask) - 1;
        mask &= mask - 1;
        if (lane == cnt) my_pos = base + bit;
        if (++cnt == tpt) {
          emit(tpt);
          cnt = 0;
          if (!alive) break;
        }
      }
    }
    if (alive && cnt > 0) emit(cnt);
    if (alive) emit(0);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      bool ok = mbar_wait(&sm.kv_full, 0, status);
      const uint32_t ka = smem_u32(sm.k), va = smem_u32(sm.v);
      const uint32_t qa = smem_u32(sm.q), da = smem_u32(sm.dout);
      const uint32_t pa = smem_u32(sm.pt), sa = smem_u32(sm.dst);
      for (int c = 0; ok; ++c) {
        ok = mbar_wait(&sm.ld_full, c & 1, status);
        if (!ok || sm.ntok == 0) break;
        tc_fence_after();
        // dP^T = V dO^T -> t_dp (free: the compute warps read it before ds_full of c-1)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma_bf16(t_dp, sdesc_sw128(va + off, 16, 1024), sdesc_sw128(da + off, 16, 1024),
                    kIdescKK, kk > 0);
        }
        // S^T = K Q^T -> t_s, once dQ^T of the previous chunk has been drained
        if (c > 0) {
          ok = mbar_wait(&sm.dq_free, (c - 1) & 1, status);
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma_bf16(t_s, sdesc_sw128(ka + off, 16, 1024), sdesc_sw128(qa + off, 16, 1024),
                    kIdescKK, kk > 0);
        }
        umma_commit(&sm.st_full);
        ok = mbar_wait(&sm.ds_full, c & 1, status);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {   // K dimension = the 128 columns
          const uint32_t aoff = (kk >> 2) * kHalf + (kk & 3) * 32;
          const uint32_t boff = kk * 2048;
          // dV += P^T dO      (A = P^T K-major, B = dO as MN-major [col][d])
          umma_bf16(t_dv, sdesc_sw128(pa + aoff, 16, 1024), sdesc_sw128(da + boff, kHalf, 1024),
                    kIdescKM, (c > 0 || kk > 0));
          // dK += dS^T Q      (A = dS^T K-major, B = Q as MN-major)
          umma_bf16(t_dk, sdesc_sw128(sa + aoff, 16, 1024), sdesc_sw128(qa + boff, kHalf, 1024),
                    kIdescKM, (c > 0 || kk > 0));
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {   // K dimension = the 128 keys
          const uint32_t off = kk * 2048;
          // dQ^T = K^T dS^T   (A = K as MN-major [key][d], B = dS^T as MN-major [key][col])
          umma_bf16(t_s, sdesc_sw128(ka + off, kHalf, 1024), sdesc_sw128(sa + off, kHalf, 1024),
                    kIdescMM, kk > 0);
        }
        umma_commit(&sm.mm_done);
        umma_commit(&sm.ld_empty);
      }
    }
  } else {
    // ------------------------------------------------------------ compute
    const int subp = warp & 3;
    const int r = subp * 32 + lane;           // key row (and head-dim row for dQ^T)
    const uint32_t trow = static_cast<uint32_t>(subp * 32) << 16;
    const int kp = b * kBlock + r;            // key position in the sequence
    const float sl2 = scale * kLog2e;
    int nchunks = 0;
    bool ok = true;
    for (int c = 0; ok; ++c) {
      if (!mbar_wait(&sm.ld_full, c & 1, status)) { ok = false; break; }
      const int ntok = sm.ntok;
      if (ntok == 0) break;
      int tokp[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) tokp[i] = (i < tpt) ? sm.tok[i] : -1;
      if (!mbar_wait(&sm.st_full, c & 1, status)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t sv[32], dv[32];
        tmem_ld32(t_s + trow + cc * 32, sv);
        tmem_ld32(t_dp + trow + cc * 32, dv);
        tmem_ld_wait();
        float pv[32], dsv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int col = cc * 32 + j;
          const int tpos = tokp[col / G];
          const bool valid = tpos >= 0 && kp <= tpos;
          const float p = valid ? exp2f(fmaf(__uint_as_float(sv[j]), sl2, -sm.lse2[col])) : 0.f;
          pv[j] = p;
          dsv[j] = p * (__uint_as_float(dv[j]) - sm.delta[col]);
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int chunk16 = cc * 4 + q4;   // 8 columns per 16-byte chunk
          const uint32_t off = (chunk16 >> 3) * kHalf + sw128_offset(r, chunk16 & 7);
          uint4 a, d;
          a.x = pack_bf16x2(pv[8 * q4 + 0], pv[8 * q4 + 1]);
          a.y = pack_bf16x2(pv[8 * q4 + 2], pv[8 * q4 + 3]);
          a.z = pack_bf16x2(pv[8 * q4 + 4], pv[8 * q4 + 5]);
          a.w = pack_bf16x2(pv[8 * q4 + 6], pv[8 * q4 + 7]);
          d.x = pack_bf16x2(dsv[8 * q4 + 0], dsv[8 * q4 + 1]);
          d.y = pack_bf16x2(dsv[8 * q4 + 2], dsv[8 * q4 + 3]);
          d.z = pack_bf16x2(dsv[8 * q4 + 4], dsv[8 * q4 + 5]);
          d.w = pack_bf16x2(dsv[8 * q4 + 6], dsv[8 * q4 + 7]);
          *reinterpret_cast<uint4*>(sm.pt + off) = a;
          *reinterpret_cast<uint4*>(sm.dst + off) = d;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.ds_full);
      // drain dQ^T (lane = head-dim channel r, column = (token, head))
      if (!mbar_wait(&sm.mm_done, c & 1, status)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t qv[32];
        tmem_ld32(t_s + trow + cc * 32, qv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int col = cc * 32 + j;
          const int ti = col / G;
          if (ti < ntok) {
            const size_t rowq = static_cast<size_t>(seq0 + tokp[ti]) * Hq + g * G + (col % G);
            atomicAdd(dq_acc + rowq * kD + r, __uint_as_float(qv[j]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.dq_free);
      ++nchunks;
    }
    // dK, dV of this item -> fp32 accumulators
    if (ok && nchunks > 0) {
      __syncwarp();
      const bool key_valid = kp < len;
      const size_t krow = (static_cast<size_t>(seq0 + kp) * Hkv + g) * kD;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t a[32], d[32];
        tmem_ld32(t_dk + trow + cc * 32, a);
        tmem_ld32(t_dv + trow + cc * 32, d);
        tmem_ld_wait();
        if (key_valid) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            atomicAdd(reinterpret_cast<float4*>(dk_acc + krow + cc * 32) + j,
                      make_float4(__uint_as_float(a[4 * j]), __uint_as_float(a[4 * j + 1]),
                                  __uint_as_float(a[4 * j + 2]), __uint_as_float(a[4 * j + 3])));
            atomicAdd(reinterpret_cast<float4*>(dv_acc + krow + cc * 32) + j,
                      make_float4(__uint_as_float(d[4 * j]), __uint_as_float(d[4 * j + 1]),
                                  __uint_as_float(d[4 * j + 2]), __uint_as_float(d[4 * j + 3])));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- host

static int bwd_max_items(int T, int S, int max_seqlen) {
  const long long max_nb = (max_seqlen + kBlock - 1) / kBlock;
  const long long tiles = plan_max_tiles(T, S);
  const long long extra = (static_cast<long long>(T) * (max_nb + 1) + 2 * kBwdSegment - 1) /
                          (2 * kBwdSegment);
  return static_cast<int>(2 * tiles + extra + 1);
}

BwdWorkspace carve_bwd_workspace(WsCursor& ws, int T, int S, int Hq, int Hkv, int max_seqlen) {
  BwdWorkspace w;
  w.plan = carve_plan(ws, T, S);
  w.max_items = bwd_max_items(T, S, max_seqlen);
  w.items = ws.take<int4>(w.max_items);
  w.num_items = ws.take<int>(1);
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
  (void)S;
  (void)max_seqlen;
  const int G = Hq / Hkv;
  if (G != 16 && G != 8)
    return fail(MSA_ERR_UNSUPPORTED, "backward supports Hq/Hkv of 8 or 16 (got %d)", G);
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t dq3[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hq),
                           static_cast<uint64_t>(T)};
  const uint64_t dkv3[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hkv),
                            static_cast<uint64_t>(T)};
  const uint32_t bq[3] = {64, static_cast<uint32_t>(G), 1};
  const uint32_t bkv[3] = {64, 1, 128};
  if (!make_tmap_bf16(&tq, q, 3, dq3, bq) || !make_tmap_bf16(&tdo, dout, 3, dq3, bq) ||
      !make_tmap_bf16(&tk, k, 3, dkv3, bkv) || !make_tmap_bf16(&tv, v, 3, dkv3, bkv))
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
    bwd_items_kernel<<<1, 1024, 0, stream>>>(cu, ws.plan.tiles, ws.plan.num_tiles, ws.items,
                                           ws.num_items, ws.max_items, st);
  }
  msa_status_t e = check_launch("bwd_delta/items");
  if (e != MSA_OK) return e;

  const size_t smem = sizeof(BwdSmem) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(sparse_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    attr_set = true;
  }
  dim3 grid(ws.max_items, Hkv);
  {
    TraceScope trace_("sparse_bwd_kernel", stream);
    sparse_bwd_kernel<<<grid, kBwdThreads, smem, stream>>>(
      tq, tk, tv, tdo, sel, cu, lse, ws.delta, ws.items, ws.num_items, Hq, Hkv, G, scale,
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
