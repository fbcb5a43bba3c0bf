// Index select: for every (token, index head) score each earlier 128-token key
// block of the token's sequence by its maximum logit q_idx . k_idx and keep the
// own block plus the 15 best earlier blocks ("MiniMax-M3.1-Flash", 1 "Model
// Introduction"; "#4581", "Kernel tuning": per-block max logits then top-k).
//
// Work unit = (128-token query tile, index head, chunk of its earlier key
// blocks).  All tokens of a tile share their own block qb, so every earlier
// block b < qb is fully causal for every row and the own block needs no score
// (it is always kept).  A plan kernel cuts each tile's blocks 0 .. qb-1 into
// chunks of at most C blocks, C chosen so that a pack yields a few units per
// SM (a pack with few long tiles is split, one with many tiles is not), and
// lists the units largest first.  The main kernel is persistent (two CTAs per
// SM, so that one's waits are covered by the other's work); warp 0 claims
// units from a counter and passes each id to the others:
//   TMA    : the unit's Q tile, then its K blocks (128 x 128 bf16, 128B
//            swizzle), each as its two 64-channel halves, into a 4-stage ring
//            of halves that runs on across units (a half is refilled once the
//            four K-steps that read it are done)
//   MMA    : S_b = Q K_b^T (M = N = K = 128) into one of two TMEM buffers
//   epilogue (4 warps, thread = query row = TMEM lane): row max of S_b; a
//            unit of at most 16 blocks keeps the maxima in a register shift
//            line and sorts them once at its end, a longer one inserts each
//            into a register-resident top-15 list as it arrives.  Both order
//            by (score descending, block id ascending): equal scores keep the
//            lower id, and an insertion moves the entries below it down in
//            order.
// A tile cut into several chunks leaves each chunk's list in the workspace;
// the chunk that finishes last (arrival counter) merges the others into its
// own in the same order and writes the selection.
// With the init rule ("#4581", Kernel tuning; read as: the first n_init
// blocks are always kept) blocks b < n_init enter the list with score +inf,
// so they take the first places and the best others fill the rest.
// The scores never leave the SM except as those 15-entry lists.
#include "kernels.cuh"

namespace msa {

namespace {

constexpr int kSelStages = 4;            // half-block stages (64 of the 128 channels)
constexpr int kSelQBufs = 1;
constexpr int kSelCtasPerSm = 2;
constexpr int kSelThreads = 192;         // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kTileBytes = 128 * 128 * 2;  // one 128 x 128 bf16 tile
constexpr int kHalfBytes = kTileBytes / 2; // its 64-channel half (one 128B-swizzled box)
constexpr uint32_t kSelIdesc = idesc_bf16(128, 128, false, false);
constexpr int kUnitSlots = 4;
constexpr int kUnitReaders = 1 + 4;      // the MMA thread and the 4 epilogue warps
constexpr int kMinChunk = 16;            // blocks
// the plan keeps the sequences' tile starts in shared memory beside its
// histogram when both fit in the default 48 KB
__host__ __device__ constexpr bool sel_plan_keeps_ts(int S, int max_nb) {
  return (max_nb + 1 + S + 1) * 4 <= 48 * 1024;
}
constexpr int kPartKeys = 15 * 128;      // one chunk's lists: entry keys, [15][128]

struct SelSmem {
  uint8_t q[kSelQBufs][kTileBytes];
  uint8_t k[kSelStages][kHalfBytes];
  uint64_t q_full[kSelQBufs], q_empty[kSelQBufs];
  uint64_t k_full[kSelStages];
  uint64_t k_empty[kSelStages];
  uint64_t s_full[2];
  uint64_t s_empty[2];
  uint64_t unit_full[kUnitSlots], unit_empty[kUnitSlots];
  int unit_id[kUnitSlots];               // claimed unit of the slot; -1: none left
  int4 unit_a[kUnitSlots];               // (sequence start, query block, first block, end block)
  int4 unit_b[kUnitSlots];               // (tile x Hi + head, chunks, first slot, chunk | rows << 16)
  uint64_t epi_sync;                     // the 4 epilogue warps (bounded waits)
  int last_flag;
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

// A list entry as one 64-bit key that orders like (score descending, block id
// ascending): the score's bits made order-preserving in the high word, the
// complement of the id in the low word (an unused entry, id -1, sorts last
// among equal scores).
__device__ __forceinline__ unsigned long long entry_key(float score, int id) {
  uint32_t u = __float_as_uint(score);
  u ^= (u & 0x80000000u) ? 0xffffffffu : 0x80000000u;
  return (static_cast<unsigned long long>(u) << 32) | (0xffffffffu - static_cast<uint32_t>(id));
}

__device__ __forceinline__ int entry_id(unsigned long long key) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(key));
}

__device__ __forceinline__ float entry_score(unsigned long long key) {
  uint32_t u = static_cast<uint32_t>(key >> 32);
  u ^= (u & 0x80000000u) ? 0x80000000u : 0xffffffffu;
  return __uint_as_float(u);
}

// k[0..15] sorted descending (bitonic sorting network)
__device__ __forceinline__ void sort16_desc(unsigned long long* k) {
#pragma unroll
  for (int w = 2; w <= 16; w <<= 1) {
#pragma unroll
    for (int j = w >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const bool desc = (i & w) == 0;
          const bool sw = desc ? (k[i] < k[l]) : (k[i] > k[l]);
          const unsigned long long a = k[i], b = k[l];
          k[i] = sw ? b : a;
          k[l] = sw ? a : b;
        }
      }
    }
  }
}

// a[0..15] and b[0..15] sorted descending -> a[0..15] = the 16 largest of
// both, sorted descending: one half-cleaner (a[i] against b[15 - i]) leaves a
// bitonic sequence holding them, which 4 merge stages sort.
__device__ __forceinline__ void merge_top16(unsigned long long* a, const unsigned long long* b) {
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = a[i] > b[15 - i] ? a[i] : b[15 - i];
#pragma unroll
  for (int j = 8; j > 0; j >>= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int l = i ^ j;
      if (l > i && a[i] < a[l]) {
        const unsigned long long t = a[i];
        a[i] = a[l];
        a[l] = t;
      }
    }
  }
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// All 128 epilogue threads meet on an mbarrier (phase `ph`, flipped here).
// Its wait is bounded like every other wait, so a warp that gave up cannot
// leave the others blocked.
__device__ __forceinline__ bool epi_sync(uint64_t* bar, uint32_t& ph, uint32_t* status) {
  mbar_arrive(bar);
  const bool ok = mbar_wait(bar, ph, status, 10);
  ph ^= 1;
  return ok;
}

// last s with tile_start[s] <= t (tile_start ascending, tile_start[0] = 0)
__device__ __forceinline__ int seq_of_tile(const int* tile_start, int S, int t) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

}  // namespace

// ---------------------------------------------------------------- plan

// One CTA.  Tiles are (sequence s, query block qb) in sequence order; tile t of
// index head h is cidx = t Hi + h.  A tile's earlier blocks are cut into
// max(1, ceil(qb / C)) chunks with C = max(16, ceil(W / kSelUnitsBeyondTiles))
// (W: all scored blocks of the pack), so that units <= tiles Hi +
// kSelUnitsBeyondTiles.  Units are listed by block count, largest first; the
// chunks of a tile cut in several get consecutive partial-list slots.  The
// counters (claim, per-tile arrivals) are cleared here for the main kernel.
__global__ void __launch_bounds__(1024) select_plan_kernel(
    const int32_t* __restrict__ cu, int S, int Hi, int max_nb, int4* __restrict__ units,
    int4* __restrict__ aux, int* __restrict__ num_units, int* __restrict__ claim,
    int* __restrict__ merge_ctr, int* __restrict__ tile_start, int max_units, int max_tiles,
    uint32_t* status) {
  pdl_enter();
  extern __shared__ int hist[];            // [max_nb + 1]: units by block count
  // tile_start[0 .. S) is searched once per (tile, head): in shared memory
  // (after hist) when it fits, else in the workspace
  int* const ts = sel_plan_keeps_ts(S, max_nb) ? hist + max_nb + 1 : tile_start;
  __shared__ int warp_sums[32];
  __shared__ int carry;
  __shared__ unsigned long long wsum;
  const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  const int nw = blockDim.x >> 5;
  for (int i = tid; i <= max_nb; i += blockDim.x) hist[i] = 0;
  if (tid == 0) {
    carry = 0;
    wsum = 0;
  }
  __syncthreads();

  // block-wide exclusive scan of v; returns the prefix (continuing from carry)
  // and advances carry by the total
  auto scan = [&](int v) -> int {
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += x;
    }
    if (lane == 31) warp_sums[wp] = incl;
    __syncthreads();
    if (wp == 0) {
      int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, w, d);
        if (lane >= d) w += x;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int off = carry + (wp > 0 ? warp_sums[wp - 1] : 0) + incl - v;
    __syncthreads();
    if (tid == blockDim.x - 1) carry = off + v;
    __syncthreads();
    return off;
  };

  // 1. tiles per sequence -> tile_start (exclusive prefix); scored blocks W
  unsigned long long wloc = 0;
  for (int base = 0; base < S; base += blockDim.x) {
    const int s = base + tid;
    int nb = 0;
    if (s < S) {
      const int len = cu[s + 1] - cu[s];
      nb = (len + kBlock - 1) / kBlock;
      if (len < 0 || nb > max_nb) {
        atomicOr(status, kStatusBounds);
        nb = len < 0 ? 0 : max_nb;
      }
      wloc += static_cast<unsigned long long>(nb) * (nb > 0 ? nb - 1 : 0) / 2;
    }
    const int off = scan(nb);
    if (s < S) ts[s] = off;
  }
  const int ntiles = min(carry, max_tiles);
  if (tid == 0 && carry > max_tiles) atomicOr(status, kStatusBounds);
  atomicAdd(&wsum, wloc);
  __syncthreads();
  const long long W = static_cast<long long>(wsum) * Hi;
  const int C = static_cast<int>(max(static_cast<long long>(kMinChunk),
                                     (W + kSelUnitsBeyondTiles - 1) / kSelUnitsBeyondTiles));

  // 2. per (tile, head): chunk count -> histogram of unit sizes
  const int ncidx = ntiles * Hi;
  for (int ci = tid; ci < ncidx; ci += blockDim.x) {
    const int t = ci / Hi;
    const int qb = t - ts[seq_of_tile(ts, S, t)];
    const int nch = qb > 0 ? (qb + C - 1) / C : 1;
    for (int c = 0; c < nch; ++c) atomicAdd(&hist[max(0, min(C, qb - c * C))], 1);
    merge_ctr[ci] = 0;
  }
  __syncthreads();
  // 3. start of each size class, largest first
  if (tid == 0) {
    int acc = 0;
    for (int z = min(C, max_nb); z >= 0; --z) {
      const int c = hist[z];
      hist[z] = acc;
      acc += c;
    }
    *num_units = min(acc, max_units);
    if (acc > max_units) atomicOr(status, kStatusBounds);
    *claim = 0;
    carry = 0;
  }
  __syncthreads();
  // 4. scatter the units; a tile cut in several chunks gets the partial slots
  //    [slot0, slot0 + nch) (exclusive prefix of those chunk counts)
  for (int base = 0; base < ncidx; base += blockDim.x) {
    const int ci = base + tid;
    int nch = 0, qb = 0, s = 0;
    if (ci < ncidx) {
      const int t = ci / Hi;
      s = seq_of_tile(ts, S, t);
      qb = t - ts[s];
      nch = qb > 0 ? (qb + C - 1) / C : 1;
    }
    const int slot0 = scan(nch > 1 ? nch : 0);
    for (int c = 0; c < nch; ++c) {
      const int b0 = c * C, b1 = min(qb, b0 + C);
      const int pos = atomicAdd(&hist[max(0, b1 - b0)], 1);
      if (pos < max_units) {
        const int seq0 = cu[s];
        const int rows = min(kBlock, cu[s + 1] - seq0 - qb * kBlock);
        units[pos] = make_int4(seq0, qb, b0, b1);
        aux[pos] = make_int4(ci, nch, slot0, c | (rows << 16));
      }
    }
  }
}

// ---------------------------------------------------------------- main kernel

__global__ void __launch_bounds__(kSelThreads, kSelCtasPerSm)
    index_select_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, const int32_t* __restrict__ cu,
                        const int4* __restrict__ units, const int4* __restrict__ aux,
                        const int* __restrict__ num_units, int* __restrict__ claim,
                        int* __restrict__ merge_ctr, unsigned long long* __restrict__ part,
                        int Hi,
                        int n_init, int32_t* __restrict__ sel, uint32_t* status) {
  pdl_enter();
  const int nunits = *num_units;
  if (static_cast<int>(blockIdx.x) >= nunits) return;
  extern __shared__ uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSelQBufs; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_empty[i], 128);
    }
    for (int i = 0; i < kSelStages; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
    }
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(&sm.unit_full[i], 1);
      mbar_init(&sm.unit_empty[i], kUnitReaders);
    }
    mbar_init(&sm.epi_sync, 128);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      // CTA i starts with unit i; later units come from the counter (unit
      // gridDim.x + claim); the next unit's record is read while this one's
      // blocks load
      int pending = blockIdx.x;
      int4 nun = units[pending], nax = aux[pending];
      uint32_t kb = 0;          // K blocks issued so far (ring position)
      uint32_t nq = 0;          // units with blocks so far (Q buffer)
      for (int ul = 0;; ++ul) {
        const int si = ul % kUnitSlots;
        const int u = pending < nunits ? pending : -1;
        const int4 un = nun, ax = nax;
        if (!mbar_wait(&sm.unit_empty[si], ((ul / kUnitSlots) & 1) ^ 1, status, 1)) break;
        sm.unit_id[si] = u;
        sm.unit_a[si] = un;
        sm.unit_b[si] = ax;
        mbar_arrive(&sm.unit_full[si]);
        if (u < 0) break;
        pending = static_cast<int>(gridDim.x) + atomicAdd(claim, 1);
        if (pending < nunits) {
          nun = units[pending];
          nax = aux[pending];
        }
        const int seq0 = un.x, qb = un.y, b0 = un.z, b1 = un.w, h = ax.x % Hi;
        if (b1 <= b0) continue;
        const int qbuf = nq % kSelQBufs;
        if (!mbar_wait(&sm.q_empty[qbuf], ((nq / kSelQBufs) & 1) ^ 1, status, 2)) break;
        ++nq;
        mbar_arrive_expect_tx(&sm.q_full[qbuf], kTileBytes);
        tma_load_3d(sm.q[qbuf], &tm_q, &sm.q_full[qbuf], 0, h, seq0 + qb * kBlock);
        tma_load_3d(sm.q[qbuf] + kHalfBytes, &tm_q, &sm.q_full[qbuf], 64, h,
                    seq0 + qb * kBlock);
        bool ok = true;
        // each K block as its two channel halves, one ring stage each: a half
        // is reloaded as soon as the four K-steps that read it are done
        for (int b = b0; ok && b < b1; ++b) {
          for (int hf = 0; hf < 2; ++hf, ++kb) {
            const int st = kb % kSelStages;
            if (!(ok = mbar_wait(&sm.k_empty[st], ((kb / kSelStages) & 1) ^ 1, status, 3))) break;
            mbar_arrive_expect_tx(&sm.k_full[st], kHalfBytes);
            tma_load_3d(sm.k[st], &tm_k, &sm.k_full[st], 64 * hf, h, seq0 + b * kBlock);
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      uint32_t kb = 0, kh = 0, nq = 0;   // blocks (S buffers), K halves (ring stages), Q tiles
      bool ok = true;
      for (int ul = 0; ok; ++ul) {
        const int si = ul % kUnitSlots;
        if (!(ok = mbar_wait(&sm.unit_full[si], (ul / kUnitSlots) & 1, status, 4))) break;
        const int u = sm.unit_id[si];
        const int4 un = sm.unit_a[si];
        mbar_arrive(&sm.unit_empty[si]);
        if (u < 0) break;
        const int nb = un.w - un.z;
        if (nb <= 0) continue;
        const int qbuf = nq % kSelQBufs;
        if (!(ok = mbar_wait(&sm.q_full[qbuf], (nq / kSelQBufs) & 1, status, 5))) break;
        ++nq;
        const uint32_t qa = smem_u32(sm.q[qbuf]);
        for (int i = 0; ok && i < nb; ++i, ++kb) {
          const int buf = kb & 1;
          if (!(ok = mbar_wait(&sm.s_empty[buf], ((kb >> 1) & 1) ^ 1, status, 7))) break;
          // channels [64 hf, 64 hf + 64): four K-steps on each half of Q and K_b
          for (int hf = 0; hf < 2; ++hf, ++kh) {
            const int st = kh % kSelStages;
            if (!(ok = mbar_wait(&sm.k_full[st], (kh / kSelStages) & 1, status, 6))) break;
            tc_fence_after();
            const uint32_t ka = smem_u32(sm.k[st]);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              umma_bf16(tmem + buf * 128, sdesc_sw128(qa + hf * kHalfBytes + kk * 32, 16, 1024),
                        sdesc_sw128(ka + kk * 32, 16, 1024), kSelIdesc, (hf | kk) != 0);
            }
            umma_commit(&sm.k_empty[st]);
          }
          if (!ok) break;
          umma_commit(&sm.s_full[buf]);
        }
        umma_commit(&sm.q_empty[qbuf]);      // the Q tile is free once these MMAs are done
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // thread = query row = TMEM lane
    const int sub = warp & 3;                 // TMEM sub-partition of this warp
    const int r = sub * 32 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    uint32_t kb = 0, eph = 0;
    for (int ul = 0;; ++ul) {
      const int si = ul % kUnitSlots;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&sm.unit_full[si], (ul / kUnitSlots) & 1, status, 8)))
        break;
      const int u = sm.unit_id[si];
      const int4 un = sm.unit_a[si];
      const int4 ax = sm.unit_b[si];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.unit_empty[si]);
      if (u < 0) break;
      const int seq0 = un.x, qb = un.y, b0 = un.z, b1 = un.w;
      const int cidx = ax.x, nch = ax.y, slot0 = ax.z, chunk = ax.w & 0xffff;
      const int nrows = ax.w >> 16;
      const int h = cidx % Hi;
      float best[15];
      int ids[15];
#pragma unroll
      for (int i = 0; i < 15; ++i) {
        best[i] = -INFINITY;
        ids[i] = -1;
      }
      bool ok = true;
      // S_b of block b -> its row max (the S buffer is freed right after the read)
      auto block_max = [&](int b) -> float {
        const int buf = kb & 1;
        ++kb;
        if (!(ok = mbar_wait(&sm.s_full[buf], ((kb - 1) >> 1) & 1, status, 9))) return 0.f;
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
        return (b < n_init) ? INFINITY : fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      };
      if (b1 - b0 <= 16) {
        // A unit of at most 16 blocks keeps every block's score in a shift
        // register (newest first) and sorts them once at its end.
        float sc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) sc[i] = -INFINITY;
        for (int b = b0; ok && b < b1; ++b) {
          const float mx = block_max(b);
#pragma unroll
          for (int i = 15; i > 0; --i) sc[i] = sc[i - 1];
          sc[0] = mx;
        }
        // sc[i] is block b1 - 1 - i; (score descending, id ascending) is the
        // order the insertion below keeps, and -inf / -1 fill unused places
        unsigned long long key[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) key[i] = (i < b1 - b0) ? entry_key(sc[i], b1 - 1 - i) : 0ull;
        sort16_desc(key);
#pragma unroll
        for (int i = 0; i < 15; ++i) {
          best[i] = key[i] ? entry_score(key[i]) : -INFINITY;
          ids[i] = key[i] ? entry_id(key[i]) : -1;
        }
      } else {
        // a longer unit inserts each block into the top-15 lists as it arrives:
        // at the first place it beats (strictly: an equal score already held
        // came from a lower block), and every later entry moves down one place
        // in order, so equal scores stay in ascending block order
        for (int b = b0; ok && b < b1; ++b) {
          float cv = block_max(b);
          int ci = b;
          bool moving = false;
#pragma unroll
          for (int i = 0; i < 15; ++i) {
            moving = moving || cv > best[i];
            if (moving) {
              const float tv = best[i];
              const int ti = ids[i];
              best[i] = cv;
              ids[i] = ci;
              cv = tv;
              ci = ti;
            }
          }
        }
      }
      // an expired wait (flagged in the status word) ends this warp's work; the
      // other warps then give up at their next bounded wait
      if (!__all_sync(0xffffffffu, ok)) break;
      bool write = true;
      if (nch > 1) {
        // leave this chunk's lists for the last chunk of the tile to finish
        unsigned long long* mine = part + static_cast<size_t>(slot0 + chunk) * kPartKeys;
#pragma unroll
        for (int i = 0; i < 15; ++i) mine[i * 128 + r] = entry_key(best[i], ids[i]);
        // the mbarrier orders the 128 threads' stores before thread 0's
        // arrival, whose release (gpu scope) publishes them with it; the last
        // chunk's acquire sees every earlier chunk's lists and passes them on
        // to its threads through the second mbarrier
        if (!epi_sync(&sm.epi_sync, eph, status)) break;
        if (r == 0) sm.last_flag = atom_add_acq_rel_gpu(merge_ctr + cidx, 1) == nch - 1;
        if (!epi_sync(&sm.epi_sync, eph, status)) break;
        write = sm.last_flag != 0;
        if (write) {
          unsigned long long key[16];
#pragma unroll
          for (int i = 0; i < 15; ++i) key[i] = entry_key(best[i], ids[i]);
          key[15] = 0ull;
          // the other chunks' lists, three at a time: all their loads are in
          // flight together, then they are merged in
          for (int c0 = 0; c0 < nch; c0 += 3) {
            unsigned long long ok16[3][16];
#pragma unroll
            for (int j = 0; j < 3; ++j) {
              const int c = c0 + j;
              const unsigned long long* other = part + static_cast<size_t>(slot0 + c) * kPartKeys;
#pragma unroll
              for (int e = 0; e < 15; ++e)
                ok16[j][e] = (c < nch && c != chunk) ? ld_relaxed_gpu(other + e * 128 + r) : 0ull;
              ok16[j][15] = 0ull;
            }
#pragma unroll
            for (int j = 0; j < 3; ++j)
              if (c0 + j < nch && c0 + j != chunk) merge_top16(key, ok16[j]);
          }
#pragma unroll
          for (int i = 0; i < 15; ++i) ids[i] = entry_id(key[i]);
        }
      }
      if (write && r < nrows)
        write_selection(sel + (static_cast<size_t>(seq0 + qb * kBlock + r) * Hi + h) * kTopK,
                        qb, ids);
      // last_flag is written again by the next split unit
      if (nch > 1 && !epi_sync(&sm.epi_sync, eph, status)) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------- host

SelWorkspace carve_select_workspace(WsCursor& ws, int T, int S, int Hi) {
  SelWorkspace w;
  w.max_tiles = plan_max_tiles(T, S);
  w.max_units = w.max_tiles * Hi + kSelUnitsBeyondTiles;
  w.units = ws.take<int4>(w.max_units);
  w.aux = ws.take<int4>(w.max_units);
  w.num_units = ws.take<int>(1);
  w.claim = ws.take<int>(1);
  w.merge_ctr = ws.take<int>(static_cast<size_t>(w.max_tiles) * Hi);
  w.tile_start = ws.take<int>(static_cast<size_t>(S) + 1);
  w.part = ws.take<unsigned long long>(static_cast<size_t>(w.max_units) * kPartKeys);
  return w;
}

msa_status_t launch_index_select(const void* q_idx, const void* k_idx, const int32_t* cu, int S,
                                 int T, int Hi, int max_seqlen, int n_init,
                                 const SelWorkspace& w, int32_t* sel, cudaStream_t stream) {
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
  const int max_nb = (max_seqlen + kBlock - 1) / kBlock;
  {
    TraceScope trace_("select_plan_kernel", stream);
    const size_t plan_smem =
        static_cast<size_t>(max_nb + 1 + (sel_plan_keeps_ts(S, max_nb) ? S + 1 : 0)) * sizeof(int);
    launch_pdl(select_plan_kernel, 1, 1024, plan_smem,
        stream, cu, S, Hi, max_nb, w.units, w.aux, w.num_units, w.claim, w.merge_ctr,
        w.tile_start, w.max_units, w.max_tiles, sw);
  }
  msa_status_t e = check_launch("select_plan_kernel");
  if (e != MSA_OK) return e;
  const int sms = device_sm_count();
  const int grid = w.max_units < kSelCtasPerSm * sms ? w.max_units : kSelCtasPerSm * sms;
  {
    TraceScope trace_("index_select_kernel", stream);
    launch_pdl(index_select_kernel, grid, kSelThreads, smem, stream, tq, tk, cu, w.units, w.aux,
        w.num_units, w.claim, w.merge_ctr, w.part, Hi, n_init, sel, sw);
  }
  return check_launch("index_select_kernel");
}

}  // namespace msa
