// Fused prologue: per-head Gemma RMSNorm, x / sqrt(mean(x^2) + eps) * (1 + w),
// followed by partial RoPE on the first 64 of 128 channels (channel i pairs
// with i + 32; angle = position * base^(-2i/64)).  ("MiniMax-M3.1-Flash",
// 1 "Model Introduction"; "MiniMax-M3" Megatron-Bridge page, "Architecture
// Notes".)  bf16 [T, H, 128] -> bf16 [T, H, 128] (in place allowed); HBM-bound.
//
// Layout of the work: a CTA takes 16 consecutive tokens of every tensor of the
// call (q, k, index q, index k: one set of angles serves them all) and sweeps
// their rows with 16 threads per row.  Thread c < 8 of a row holds channels
// [4c, 4c + 4) and [4c + 32, 4c + 36): the rotated pairs (i, i + 32) sit in one
// thread, so the rotation needs no shuffles; threads 8..15 hold the
// pass-through channels 64..127.  Each thread keeps four rows in registers:
// three rows' loads are in flight while the fourth is processed, and the first
// rows' loads are issued before the angles are computed.
//
// Angles avoid a large fp32 argument: the host turns each frequency f_i into
// the 64-bit fixed-point fraction F_i = f_i / (2 pi) * 2^64 of a turn, so
// position * F_i (mod 2^64, plain integer wrap-around) is the exact angle in
// turns; its signed value times 2^-63 is the angle / pi in [-1, 1), which
// sincospif evaluates.
#include <cmath>
#include "kernels.cuh"

namespace msa {

struct RopeTurns {
  unsigned long long f[kRopeDim / 2];
};

struct PrologueArgs {
  PrologueJob jobs[4];
  int hstart[5];
};

constexpr int kProTokens = 16;
constexpr int kProThreads = 256;             // decode-append kernel
constexpr int kProSlots = kProThreads / 8;   // rows processed side by side
// forward kernel: 128 threads, 8 rows side by side with 16 threads per row
// (8 channels each: thread c < 8 holds the rotated pairs (4c + e, 4c + 32 + e),
// c >= 8 the pass-through channels 64 + 8 (c - 8) ..); four rows per thread in
// registers, so three rows' loads are in flight while the fourth is
// normalised, rotated and stored (62 registers, 8 CTAs per SM)
constexpr int kPfThreads = 128;
constexpr int kPfLanes = 16;
constexpr int kPfSlots = kPfThreads / kPfLanes;

__global__ void __launch_bounds__(kPfThreads, 8) prologue_kernel(const PrologueArgs args,
                                                                  const RopeTurns turns,
                                                                  const int32_t* __restrict__ cu,
                                                                  int S, int T, float eps,
                                                                  uint32_t* status) {
  pdl_enter();
  __shared__ float2 cs[kProTokens][kRopeDim / 2];
  __shared__ __align__(16) float wsh[4][kD];
  const int t0 = blockIdx.x * kProTokens;
  const int tid = threadIdx.x;
  const int hsum = args.hstart[4];
  const int c = tid & (kPfLanes - 1);     // channel group of the row
  const int slot = tid / kPfLanes;
  // channel offsets (elements) of this thread's two 4-channel pieces
  const int off0 = (c < 8) ? 4 * c : 64 + 8 * (c - 8);
  const int off1 = (c < 8) ? 4 * c + 32 : 64 + 8 * (c - 8) + 4;
  // 1 + w of every job (read after the barrier below)
  for (int k = tid; k < 4 * kD; k += blockDim.x) {
    const int j = k / kD;
    wsh[j][k % kD] = (args.hstart[j] < args.hstart[j + 1])
                         ? 1.f + __bfloat162float(args.jobs[j].w[k % kD]) : 0.f;
  }
  const int ntok = min(kProTokens, T - t0);
  const int rows = ntok * hsum;

  // This thread's rows are slot, slot + 8, slot + 16, ...; (tl, k) = (token of
  // the CTA, row within the token) advances by 8 rows per step without a
  // division once hsum is known.
  int tl = slot / hsum, k = slot - (slot / hsum) * hsum;
  auto advance = [&]() {
    k += kPfSlots;
    while (k >= hsum) {
      k -= hsum;
      ++tl;
    }
  };
  struct Rows {
    uint2 xa, xb;
    int rj, rtl;
    size_t rrow;
  };
  Rows ra, rb, rc, rd;
  // loads the thread's next row (rows are taken in order; r = the row index)
  auto load_rows = [&](int r, Rows& R) {
    R.rj = -1;
    R.rtl = 0;
    R.rrow = 0;
    R.xa = make_uint2(0, 0);
    R.xb = R.xa;
    if (r < rows) {
      const int j = (k >= args.hstart[1]) + (k >= args.hstart[2]) + (k >= args.hstart[3]);
      const size_t row = static_cast<size_t>(t0 + tl) * args.jobs[j].H + (k - args.hstart[j]);
      const __nv_bfloat16* src = args.jobs[j].x + row * kD;
      R.xa = __ldcs(reinterpret_cast<const uint2*>(src + off0));
      R.xb = __ldcs(reinterpret_cast<const uint2*>(src + off1));
      R.rj = j;
      R.rtl = tl;
      R.rrow = row;
      advance();
    }
  };
  // the first rows' loads are in flight while the angles are computed
  load_rows(slot, ra);
  load_rows(kPfSlots + slot, rb);
  load_rows(2 * kPfSlots + slot, rc);
  // (cos, sin) for the CTA's tokens: thread = (token, frequency)
  for (int q = tid; q < kProTokens * (kRopeDim / 2); q += blockDim.x) {
    const int qt = q / (kRopeDim / 2), i = q % (kRopeDim / 2);
    const int t = t0 + qt;
    float cv = 1.f, sv = 0.f;
    if (t < T) {
      int lo = 0, hi = S;   // largest s with cu[s] <= t
      while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
      }
      const unsigned long long pos = static_cast<unsigned long long>(t - __ldg(cu + lo));
      const long long ang = static_cast<long long>(pos * turns.f[i]);
      const float x = static_cast<float>(ang) * 1.0842021724855044e-19f;   // * 2^-63
      sincospif(x, &sv, &cv);
    }
    cs[qt][i] = make_float2(cv, sv);
  }
  __syncthreads();

  auto process = [&](const Rows& R) {
    float x[8];
    {
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&R.xa);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&R.xb);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float2 fa = __bfloat1622float2(pa[e]);
        const float2 fb = __bfloat1622float2(pb[e]);
        x[2 * e] = fa.x;
        x[2 * e + 1] = fa.y;
        x[4 + 2 * e] = fb.x;
        x[4 + 2 * e + 1] = fb.y;
      }
    }
    float s2[2] = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 8; ++e) s2[e & 1] = fmaf(x[e], x[e], s2[e & 1]);
    float ss = s2[0] + s2[1];
#pragma unroll
    for (int m = kPfLanes / 2; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const int j = R.rj < 0 ? 0 : R.rj;
    const float rinv = rsqrtf(ss * (1.f / kD) + eps);
    {
      const float4 w0 = *reinterpret_cast<const float4*>(&wsh[j][off0]);
      const float4 w1 = *reinterpret_cast<const float4*>(&wsh[j][off1]);
      const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= rinv * w[e];
    }
    if (c < 8) {
      // rotate channel 4c + e (x1) with 4c + 32 + e (x2), frequency 4c + e
      const float4* cp = reinterpret_cast<const float4*>(&cs[R.rtl][4 * c]);
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const float4 q = cp[e2];   // (cos, sin) of frequencies 2 e2, 2 e2 + 1
        const float cc[2] = {q.x, q.z}, sn[2] = {q.y, q.w};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int e = 2 * e2 + h;
          const float x1 = x[e], x2 = x[4 + e];
          x[e] = x1 * cc[h] - x2 * sn[h];
          x[4 + e] = x2 * cc[h] + x1 * sn[h];
        }
      }
    }
    if (R.rj >= 0) {
      uint2 oa, ob;
      oa.x = pack_bf16x2(x[0], x[1]);
      oa.y = pack_bf16x2(x[2], x[3]);
      ob.x = pack_bf16x2(x[4], x[5]);
      ob.y = pack_bf16x2(x[6], x[7]);
      __nv_bfloat16* dst = args.jobs[R.rj].y + R.rrow * kD;
      *reinterpret_cast<uint2*>(dst + off0) = oa;
      *reinterpret_cast<uint2*>(dst + off1) = ob;
    }
  };
  // the loop bound is uniform over the CTA: every lane reaches the shuffles;
  // three rows' loads are in flight while the fourth row is processed
  for (int base = 0; base < rows; base += 4 * kPfSlots) {
    load_rows(base + 3 * kPfSlots + slot, rd);
    process(ra);
    if (base + kPfSlots >= rows) break;
    load_rows(base + 4 * kPfSlots + slot, ra);
    process(rb);
    if (base + 2 * kPfSlots >= rows) break;
    load_rows(base + 5 * kPfSlots + slot, rb);
    process(rc);
    if (base + 3 * kPfSlots >= rows) break;
    load_rows(base + 6 * kPfSlots + slot, rc);
    process(rd);
  }
}

msa_status_t launch_prologue(const PrologueJob* jobs, int njobs, const int32_t* cu, int S, int T,
                             float rope_base, float eps, cudaStream_t stream) {
  if (njobs < 1 || njobs > 4) return fail(MSA_ERR_INVALID_ARG, "prologue takes 1..4 tensors");
  PrologueArgs args{};
  int h = 0;
  for (int j = 0; j < 4; ++j) {
    args.hstart[j] = h;
    if (j < njobs) { args.jobs[j] = jobs[j]; h += jobs[j].H; }
    else { args.jobs[j] = jobs[0]; args.jobs[j].H = 0; }
  }
  args.hstart[4] = h;
  RopeTurns turns;
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < kRopeDim / 2; ++i) {
    double f = std::pow(static_cast<double>(rope_base), -2.0 * i / kRopeDim);
    turns.f[i] = static_cast<unsigned long long>(f / two_pi * 18446744073709551616.0);
  }
  uint32_t* sw = nullptr;
  if (msa_status_t e_ = status_word(&sw); e_ != MSA_OK) return e_;
  dim3 grid((T + kProTokens - 1) / kProTokens);
  {
    TraceScope trace_("prologue_kernel", stream);
    launch_pdl(prologue_kernel, grid, kPfThreads, 0, stream, args, turns, cu, S, T, eps,
        sw);
  }
  return check_launch("prologue_kernel");
}

// ---------------------------------------------------------------- backward
//
// Gradients of the prologue of one tensor: given dy = dL/dy [T, H, 128],
// dx = dL/dx (bf16, same layout) and dw = dL/dw (fp32 [128], summed over
// tokens and heads).  RoPE is a rotation, so dz = R^T dy (the pairs turned back
// by the angle); with r = rsqrt(mean(x^2) + eps), xh = x r, g = dz (1 + w):
//   dx = r (g - xh mean(g xh)),   dw = sum dz xh.
// A CTA takes one group of 16 tokens (CTAs take several groups when there are
// more than 2048) with 128 threads: 8 rows side by side, 16 threads per row
// holding 8 channels each (thread c < 8: the rotated pairs (4c + e,
// 4c + 32 + e); c >= 8: the pass-through channels 64 + 8 (c - 8) ..).  Each
// thread keeps three rows in registers: two rows' loads are in flight while
// the third is processed.  Few live values per thread keep 7 CTAs on an SM.
// Each thread sums dw for its 8 channels over its rows, the CTA adds its 8 row
// slots into one partial row of dw_part, and prologue_bwd_sum_kernel adds the
// partials in a fixed order (the result does not depend on scheduling).
constexpr int kPbThreads = 128;
constexpr int kPbLanes = 16;                 // threads per row
constexpr int kPbSlots = kPbThreads / kPbLanes;

__global__ void __launch_bounds__(kPbThreads, 7) prologue_bwd_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ dy,
    __nv_bfloat16* __restrict__ dx, const __nv_bfloat16* __restrict__ w, int H,
    const RopeTurns turns, const int32_t* __restrict__ cu, int S, int T, float eps,
    float* __restrict__ dw_part) {
  pdl_enter();
  __shared__ float2 cs[kProTokens][kRopeDim / 2];
  __shared__ __align__(16) float wsh[kD];
  __shared__ float red[kPbSlots][kD + 4];
  const int tid = threadIdx.x;
  const int c = tid & (kPbLanes - 1);
  const int slot = tid / kPbLanes;
  const int off0 = (c < 8) ? 4 * c : 64 + 8 * (c - 8);
  const int off1 = (c < 8) ? 4 * c + 32 : 64 + 8 * (c - 8) + 4;
  for (int k = tid; k < kD; k += blockDim.x) wsh[k] = 1.f + __bfloat162float(w[k]);
  float aw[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) aw[e] = 0.f;
  struct Rows {
    uint2 xa, xb, ga, gb;
    int r;                                 // row of the group, -1: none
  };
  const int ngroups = (T + kProTokens - 1) / kProTokens;
  // grid-stride over groups of 16 tokens; dw accumulates across all of them
  for (int grp = blockIdx.x; grp < ngroups; grp += gridDim.x) {
    const int t0 = grp * kProTokens;
    const int ntok = min(kProTokens, T - t0);
    const int rows = ntok * H;
    const size_t row_base = static_cast<size_t>(t0) * H;   // the CTA's rows are contiguous
    auto load_rows = [&](int r, Rows& R) {
      R.r = -1;
      R.xa = R.xb = R.ga = R.gb = make_uint2(0, 0);
      if (r < rows) {
        const __nv_bfloat16* xr = x + (row_base + r) * kD;
        const __nv_bfloat16* gr = dy + (row_base + r) * kD;
        R.xa = __ldcs(reinterpret_cast<const uint2*>(xr + off0));
        R.xb = __ldcs(reinterpret_cast<const uint2*>(xr + off1));
        R.ga = __ldcs(reinterpret_cast<const uint2*>(gr + off0));
        R.gb = __ldcs(reinterpret_cast<const uint2*>(gr + off1));
        R.r = r;
      }
    };
    Rows ra, rb, rc, rd;
    __syncthreads();                       // the previous group's angles are consumed
    load_rows(slot, ra);                   // in flight while the angles are computed
    load_rows(kPbSlots + slot, rb);
    for (int q = tid; q < kProTokens * (kRopeDim / 2); q += blockDim.x) {
      const int qt = q / (kRopeDim / 2), i = q % (kRopeDim / 2);
      const int t = t0 + qt;
      float cv = 1.f, sv = 0.f;
      if (t < T) {
        int lo = 0, hi = S;   // largest s with cu[s] <= t
        while (hi - lo > 1) {
          int mid = (lo + hi) >> 1;
          if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
        }
        const unsigned long long pos = static_cast<unsigned long long>(t - __ldg(cu + lo));
        const long long ang = static_cast<long long>(pos * turns.f[i]);
        const float a = static_cast<float>(ang) * 1.0842021724855044e-19f;   // * 2^-63
        sincospif(a, &sv, &cv);
      }
      cs[qt][i] = make_float2(cv, sv);
    }
    __syncthreads();

    auto process = [&](const Rows& R) {
      const bool valid = R.r >= 0;
      const int tl = valid ? R.r / H : 0;
      float xv[8], dz[8];
      {
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&R.xa);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&R.xb);
        const __nv_bfloat162* qa = reinterpret_cast<const __nv_bfloat162*>(&R.ga);
        const __nv_bfloat162* qb = reinterpret_cast<const __nv_bfloat162*>(&R.gb);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float2 fa = __bfloat1622float2(pa[e]), fb = __bfloat1622float2(pb[e]);
          const float2 da = __bfloat1622float2(qa[e]), db = __bfloat1622float2(qb[e]);
          xv[2 * e] = fa.x;
          xv[2 * e + 1] = fa.y;
          xv[4 + 2 * e] = fb.x;
          xv[4 + 2 * e + 1] = fb.y;
          dz[2 * e] = da.x;
          dz[2 * e + 1] = da.y;
          dz[4 + 2 * e] = db.x;
          dz[4 + 2 * e + 1] = db.y;
        }
      }
      if (c < 8) {
        // dz = R^T dy for the pairs (4c + e, 4c + 32 + e), frequency 4c + e
        const float4* cp = reinterpret_cast<const float4*>(&cs[tl][4 * c]);
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const float4 q4 = cp[e2];
          const float cc[2] = {q4.x, q4.z}, sn[2] = {q4.y, q4.w};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int e = 2 * e2 + h;
            const float d1 = dz[e], d2 = dz[4 + e];
            dz[e] = d1 * cc[h] + d2 * sn[h];
            dz[4 + e] = d2 * cc[h] - d1 * sn[h];
          }
        }
      }
      float s2[2] = {0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 8; ++e) s2[e & 1] = fmaf(xv[e], xv[e], s2[e & 1]);
      float ss = s2[0] + s2[1];
#pragma unroll
      for (int m = kPbLanes / 2; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      const float rinv = rsqrtf(ss * (1.f / kD) + eps);
      float gw[8];
      {
        const float4 w0 = *reinterpret_cast<const float4*>(&wsh[off0]);
        const float4 w1 = *reinterpret_cast<const float4*>(&wsh[off1]);
        gw[0] = w0.x; gw[1] = w0.y; gw[2] = w0.z; gw[3] = w0.w;
        gw[4] = w1.x; gw[5] = w1.y; gw[6] = w1.z; gw[7] = w1.w;
      }
      float d2[2] = {0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        xv[e] *= rinv;                     // xh
        gw[e] *= dz[e];                    // g = dz (1 + w)
        d2[e & 1] = fmaf(gw[e], xv[e], d2[e & 1]);
      }
      float dot = d2[0] + d2[1];
#pragma unroll
      for (int m = kPbLanes / 2; m >= 1; m >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, m);
      const float mean = dot * (1.f / kD);
      if (valid) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          o[e] = rinv * (gw[e] - xv[e] * mean);
          aw[e] = fmaf(dz[e], xv[e], aw[e]);
        }
        uint2 oa, ob;
        oa.x = pack_bf16x2(o[0], o[1]);
        oa.y = pack_bf16x2(o[2], o[3]);
        ob.x = pack_bf16x2(o[4], o[5]);
        ob.y = pack_bf16x2(o[6], o[7]);
        __nv_bfloat16* dr = dx + (row_base + R.r) * kD;
        *reinterpret_cast<uint2*>(dr + off0) = oa;
        *reinterpret_cast<uint2*>(dr + off1) = ob;
      }
    };
    // the loop bound is uniform over the CTA: every lane reaches the shuffles;
    // two rows' loads are in flight while the third row is processed
    for (int base = 0; base < rows; base += 3 * kPbSlots) {
      load_rows(base + 2 * kPbSlots + slot, rc);
      process(ra);
      if (base + kPbSlots >= rows) break;
      load_rows(base + 3 * kPbSlots + slot, ra);
      process(rb);
      if (base + 2 * kPbSlots >= rows) break;
      load_rows(base + 4 * kPbSlots + slot, rb);
      process(rc);
    }
  }
  // ---- dw: the CTA's 8 row slots -> one partial row
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    red[slot][off0 + e] = aw[e];
    red[slot][off1 + e] = aw[4 + e];
  }
  __syncthreads();
  for (int ch = tid; ch < kD; ch += blockDim.x) {
    float acc = 0.f;
    for (int sl = 0; sl < kPbSlots; ++sl) acc += red[sl][ch];
    dw_part[static_cast<size_t>(blockIdx.x) * kD + ch] = acc;
  }
}

// dw[ch] = sum over the partial rows in a fixed order (the result does not
// depend on scheduling): CTA b takes channels 8b .. 8b + 7 with 1024 threads,
// thread (k, ch) adds the partials k, k + 128, ... of its channel, then a
// pairwise tree over k in shared memory.
constexpr int kPbSumChannels = 8;
constexpr int kPbSumWays = 1024 / kPbSumChannels;
__global__ void __launch_bounds__(1024) prologue_bwd_sum_kernel(const float* __restrict__ part,
                                                                int nparts,
                                                                float* __restrict__ dw) {
  pdl_enter();
  __shared__ float red[kPbSumWays][kPbSumChannels];
  const int cl = threadIdx.x % kPbSumChannels, k = threadIdx.x / kPbSumChannels;
  const int ch = blockIdx.x * kPbSumChannels + cl;
  float acc = 0.f;
  for (int p = k; p < nparts; p += kPbSumWays) acc += part[static_cast<size_t>(p) * kD + ch];
  red[k][cl] = acc;
  __syncthreads();
#pragma unroll
  for (int s = kPbSumWays / 2; s >= 1; s >>= 1) {
    if (k < s) red[k][cl] += red[k + s][cl];
    __syncthreads();
  }
  if (k == 0) dw[ch] = red[0][cl];
}

constexpr int kProBwdMaxCtas = 2048;   // partial rows at most

// one CTA per group of 16 tokens up to 2048 groups (32k tokens), then CTAs
// take several groups each
static int prologue_bwd_ctas(int T) {
  const int groups = (T + kProTokens - 1) / kProTokens;
  return groups < kProBwdMaxCtas ? groups : kProBwdMaxCtas;
}

size_t prologue_bwd_workspace_floats(int T) {
  const int groups = (T + kProTokens - 1) / kProTokens;
  return static_cast<size_t>(groups < kProBwdMaxCtas ? groups : kProBwdMaxCtas) * kD;
}

msa_status_t launch_prologue_bwd(const __nv_bfloat16* x, const __nv_bfloat16* dy,
                                 __nv_bfloat16* dx, float* dw, const __nv_bfloat16* w, int H,
                                 const int32_t* cu, int S, int T, float rope_base, float eps,
                                 float* dw_part, cudaStream_t stream) {
  RopeTurns turns;
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < kRopeDim / 2; ++i) {
    double f = std::pow(static_cast<double>(rope_base), -2.0 * i / kRopeDim);
    turns.f[i] = static_cast<unsigned long long>(f / two_pi * 18446744073709551616.0);
  }
  const int nparts = prologue_bwd_ctas(T);
  {
    TraceScope trace_("prologue_bwd_kernel", stream);
    launch_pdl(prologue_bwd_kernel, nparts, kPbThreads, 0, stream, x, dy, dx, w, H, turns, cu, S, T,
        eps, dw_part);
  }
  msa_status_t e = check_launch("prologue_bwd_kernel");
  if (e != MSA_OK) return e;
  {
    TraceScope trace_("prologue_bwd_sum_kernel", stream);
    launch_pdl(prologue_bwd_sum_kernel, kD / kPbSumChannels, 1024, 0, stream, dw_part, nparts, dw);
  }
  return check_launch("prologue_bwd_sum_kernel");
}

// ---------------------------------------------------------------- decode append
//
// One new token per sequence b at position p = cache_lens[b] - 1: the prologue
// of its q and index-q (to q_out, q_idx_out) and of its k and index-k, which
// go with its v (unchanged) into slot p % 128 of page block_table[b, p / 128].
// Grid (B, row chunks): a CTA takes 32 of sequence b's rows, 8 threads per row
// as in the prologue kernels.  Row order: q (Hq), index-q (H), k (H),
// index-k (H), v (H), H = Hkv.

struct AppendArgs {
  const __nv_bfloat16* src[5];    // q, q_idx, k, k_idx, v  [B, heads, 128]
  const __nv_bfloat16* w[4];      // w_q, w_qi, w_k, w_ki
  __nv_bfloat16* q_out;
  __nv_bfloat16* qi_out;
  __nv_bfloat16* cache[3];        // k, k_idx, v caches [page, H, 128 slots, 128]
  int Hq, H;
};

__global__ void __launch_bounds__(kProThreads) decode_append_kernel(
    const AppendArgs a, const RopeTurns turns, const int32_t* __restrict__ block_table,
    const int32_t* __restrict__ cache_lens, int num_pages, int max_pages, float eps,
    uint32_t* status) {
  pdl_enter();
  __shared__ float2 cs[kRopeDim / 2];
  __shared__ float wsh[4][kD];
  const int b = blockIdx.x, tid = threadIdx.x;
  const int L = cache_lens[b];
  if (L < 1 || L > max_pages * kBlock) {
    if (tid == 0 && blockIdx.y == 0) atomicOr(status, kStatusBounds);
    return;
  }
  const int p = L - 1;
  const int page = block_table[static_cast<size_t>(b) * max_pages + p / kBlock];
  if (page < 0 || page >= num_pages) {
    if (tid == 0 && blockIdx.y == 0) atomicOr(status, kStatusBounds);
    return;
  }
  const int slot_in_page = p % kBlock;
  for (int k = tid; k < 4 * kD; k += blockDim.x) {
    const int j = k / kD;
    const __nv_bfloat16* wp = (j == 0) ? a.w[0] : (j == 1) ? a.w[1] : (j == 2) ? a.w[2] : a.w[3];
    wsh[j][k % kD] = 1.f + __bfloat162float(wp[k % kD]);
  }
  if (tid < kRopeDim / 2) {
    const long long ang = static_cast<long long>(static_cast<unsigned long long>(p) * turns.f[tid]);
    float cv, sv;
    sincospif(static_cast<float>(ang) * 1.0842021724855044e-19f, &sv, &cv);   // * 2^-63
    cs[tid] = make_float2(cv, sv);
  }
  __syncthreads();
  const int c = tid & 7, rs = tid >> 3;
  const int off0 = (c < 4) ? 8 * c : 64 + 16 * (c - 4);
  const int off1 = (c < 4) ? 8 * c + 32 : 64 + 16 * (c - 4) + 8;
  const int H = a.H, Hq = a.Hq;
  const int rows = Hq + 4 * H;
  // the loop bound is uniform over the CTA: every lane reaches the shuffles
  for (int base = blockIdx.y * kProSlots; base < rows; base += gridDim.y * kProSlots) {
    const int r = base + rs;
    const bool valid = r < rows;
    // job: 0 q, 1 index-q, 2 k, 3 index-k, 4 v
    int job = 0, h = r;
    if (r >= Hq) {
      job = 1 + (r - Hq) / H;
      h = (r - Hq) % H;
    }
    if (!valid) job = 0, h = 0;
    const int heads = (job == 0) ? Hq : H;
    const __nv_bfloat16* sbase = (job == 0) ? a.src[0] : (job == 1) ? a.src[1]
                               : (job == 2) ? a.src[2] : (job == 3) ? a.src[3] : a.src[4];
    const __nv_bfloat16* src = sbase + (static_cast<size_t>(b) * heads + h) * kD;
    uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
    if (valid) {
      xa = *reinterpret_cast<const uint4*>(src + off0);
      xb = *reinterpret_cast<const uint4*>(src + off1);
    }
    __nv_bfloat16* dst;
    if (job <= 1) {
      dst = (job == 0 ? a.q_out : a.qi_out) + (static_cast<size_t>(b) * heads + h) * kD;
    } else {
      __nv_bfloat16* cbase = (job == 2) ? a.cache[0] : (job == 3) ? a.cache[1] : a.cache[2];
      dst = cbase + ((static_cast<size_t>(page) * H + h) * kBlock + slot_in_page) * kD;
    }
    if (job == 4) {                        // v: stored as given
      if (valid) {
        *reinterpret_cast<uint4*>(dst + off0) = xa;
        *reinterpret_cast<uint4*>(dst + off1) = xb;
      }
      continue;
    }
    float x[16];
    {
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&xa);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&xb);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(pa[e]);
        const float2 fb = __bfloat1622float2(pb[e]);
        x[2 * e] = fa.x;
        x[2 * e + 1] = fa.y;
        x[8 + 2 * e] = fb.x;
        x[8 + 2 * e + 1] = fb.y;
      }
    }
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 16; ++e) s4[e & 3] = fmaf(x[e], x[e], s4[e & 3]);
    float ss = (s4[0] + s4[1]) + (s4[2] + s4[3]);
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const float rinv = rsqrtf(ss * (1.f / kD) + eps);
    const int wj = (job == 0) ? 0 : (job == 1) ? 1 : (job == 2) ? 2 : 3;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      x[e] *= rinv * wsh[wj][off0 + e];
      x[8 + e] *= rinv * wsh[wj][off1 + e];
    }
    if (c < 4) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 q = cs[8 * c + e];
        const float x1 = x[e], x2 = x[8 + e];
        x[e] = x1 * q.x - x2 * q.y;
        x[8 + e] = x2 * q.x + x1 * q.y;
      }
    }
    if (valid) {
      uint4 oa, ob;
      oa.x = pack_bf16x2(x[0], x[1]);
      oa.y = pack_bf16x2(x[2], x[3]);
      oa.z = pack_bf16x2(x[4], x[5]);
      oa.w = pack_bf16x2(x[6], x[7]);
      ob.x = pack_bf16x2(x[8], x[9]);
      ob.y = pack_bf16x2(x[10], x[11]);
      ob.z = pack_bf16x2(x[12], x[13]);
      ob.w = pack_bf16x2(x[14], x[15]);
      *reinterpret_cast<uint4*>(dst + off0) = oa;
      *reinterpret_cast<uint4*>(dst + off1) = ob;
    }
  }
}

msa_status_t launch_decode_append(const DecodeAppendJob& j, const int32_t* block_table,
                                  const int32_t* cache_lens, int B, int num_pages,
                                  int max_pages, float rope_base, float eps,
                                  cudaStream_t stream) {
  AppendArgs a;
  a.src[0] = j.q;
  a.src[1] = j.q_idx;
  a.src[2] = j.k;
  a.src[3] = j.k_idx;
  a.src[4] = j.v;
  a.w[0] = j.w_q;
  a.w[1] = j.w_qi;
  a.w[2] = j.w_k;
  a.w[3] = j.w_ki;
  a.q_out = j.q_out;
  a.qi_out = j.q_idx_out;
  a.cache[0] = j.k_cache;
  a.cache[1] = j.kidx_cache;
  a.cache[2] = j.v_cache;
  a.Hq = j.Hq;
  a.H = j.Hkv;
  RopeTurns turns;
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < kRopeDim / 2; ++i) {
    double f = std::pow(static_cast<double>(rope_base), -2.0 * i / kRopeDim);
    turns.f[i] = static_cast<unsigned long long>(f / two_pi * 18446744073709551616.0);
  }
  uint32_t* sw = nullptr;
  if (msa_status_t e_ = status_word(&sw); e_ != MSA_OK) return e_;
  {
    TraceScope trace_("decode_append_kernel", stream);
    dim3 grid(B, (j.Hq + 4 * j.Hkv + kProSlots - 1) / kProSlots);
    launch_pdl(decode_append_kernel, grid, kProThreads, 0, stream, a, turns, block_table, cache_lens,
        num_pages, max_pages, eps,
        sw);
  }
  return check_launch("decode_append_kernel");
}

}  // namespace msa
