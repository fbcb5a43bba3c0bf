// Fused prologue: per-head Gemma RMSNorm, x / sqrt(mean(x^2) + eps) * (1 + w),
// followed by partial RoPE on the first 64 of 128 channels (channel i pairs
// with i + 32; angle = position * base^(-2i/64)).  ("MiniMax-M3.1-Flash",
// 1 "Model Introduction"; "MiniMax-M3" Megatron-Bridge page, "Architecture
// Notes".)  bf16 [T, H, 128] -> bf16 [T, H, 128] (in place allowed); HBM-bound.
//
// Layout of the work: a CTA takes 16 consecutive tokens of every tensor of the
// call (q, k, index q, index k: one set of angles serves them all).  It first
// issues the loads of its first 128 rows (8 per thread), computes the 16 x 32
// (cos, sin) pairs of its tokens meanwhile, then sweeps the rows, 16 threads
// per row and 8 channels (16 bytes) per thread.
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
constexpr int kProUnroll = 8;      // rows per thread per sweep step (loads in flight)

__global__ void __launch_bounds__(256, 4) prologue_kernel(const PrologueArgs args,
                                                       const RopeTurns turns,
                                                       const int32_t* __restrict__ cu, int S,
                                                       int T, float eps, uint32_t* status) {
  __shared__ float2 cs[kProTokens][kRopeDim / 2];
  __shared__ float wsh[4][kD];
  const int t0 = blockIdx.x * kProTokens;
  const int tid = threadIdx.x;
  const int hsum = args.hstart[4];
  // 1 + w of every job (read after the barrier below)
  for (int k = tid; k < 4 * kD; k += blockDim.x) {
    const int j = k / kD;
    wsh[j][k % kD] = (args.hstart[j] < args.hstart[j + 1])
                         ? 1.f + __bfloat162float(args.jobs[j].w[k % kD]) : 0.f;
  }
  const int chunk = tid & 15;           // 8 channels: [8 chunk, 8 chunk + 8)
  const int ntok = min(kProTokens, T - t0);
  const int rows = ntok * hsum;
  uint4 xv[kProUnroll];
  // sweep row r of the CTA -> job j, row of that tensor, token of the CTA
  auto row_of = [&](int r, int& j, size_t& row, int& tl) {
    tl = r / hsum;
    const int k = r - tl * hsum;
    j = (k >= args.hstart[1]) + (k >= args.hstart[2]) + (k >= args.hstart[3]);
    row = static_cast<size_t>(t0 + tl) * args.jobs[j].H + (k - args.hstart[j]);
  };
  auto load_rows = [&](int base) {
#pragma unroll
    for (int u = 0; u < kProUnroll; ++u) {
      const int r = base + (tid >> 4) + 16 * u;
      xv[u] = make_uint4(0, 0, 0, 0);
      if (r < rows) {
        int j, tl; size_t row;
        row_of(r, j, row, tl);
        xv[u] = __ldcs(reinterpret_cast<const uint4*>(args.jobs[j].x + row * kD) + chunk);
      }
    }
  };
  load_rows(0);   // in flight while the angles are computed
  // (cos, sin) for the CTA's tokens: thread = (token, frequency)
  for (int k = tid; k < kProTokens * (kRopeDim / 2); k += blockDim.x) {
    const int tl = k / (kRopeDim / 2), i = k % (kRopeDim / 2);
    const int t = t0 + tl;
    float c = 1.f, s = 0.f;
    if (t < T) {
      int lo = 0, hi = S;   // largest s with cu[s] <= t
      while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
      }
      const unsigned long long pos = static_cast<unsigned long long>(t - __ldg(cu + lo));
      const long long ang = static_cast<long long>(pos * turns.f[i]);
      const float x = static_cast<float>(ang) * 1.0842021724855044e-19f;   // * 2^-63
      sincospif(x, &s, &c);
    }
    cs[tl][i] = make_float2(c, s);
  }
  __syncthreads();
  // the loop bound is uniform over the CTA: every lane reaches the shuffles
  for (int base = 0; base < rows; base += 16 * kProUnroll) {
    if (base > 0) load_rows(base);
#pragma unroll
    for (int u = 0; u < kProUnroll; ++u) {
      const int r = base + (tid >> 4) + 16 * u;
      int j = 0, tl = 0; size_t row = 0;
      if (r < rows) row_of(r, j, row, tl);
      float x[8];
      {
        const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&xv[u]);
#pragma unroll
        for (int e = 0; e < 4; ++e) { float2 f = __bfloat1622float2(xp[e]); x[2 * e] = f.x; x[2 * e + 1] = f.y; }
      }
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
      for (int m = 8; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      const float rinv = rsqrtf(ss * (1.f / kD) + eps);
      const float4 w0 = *reinterpret_cast<const float4*>(&wsh[j][8 * chunk]);
      const float4 w1 = *reinterpret_cast<const float4*>(&wsh[j][8 * chunk + 4]);
      const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = x[e] * rinv * w[e];
      // rotate-half on channels [0, 64): chunk c < 4 holds x1, chunk c + 4 holds x2
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = __shfl_xor_sync(0xffffffffu, x[e], 4);
      if (chunk < 8) {
        const int fbase = (chunk & 3) * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 c = cs[tl][fbase + e];
          x[e] = (chunk < 4) ? (x[e] * c.x - y[e] * c.y) : (x[e] * c.x + y[e] * c.y);
        }
      }
      if (r < rows) {
        uint4 out;
        out.x = pack_bf16x2(x[0], x[1]); out.y = pack_bf16x2(x[2], x[3]);
        out.z = pack_bf16x2(x[4], x[5]); out.w = pack_bf16x2(x[6], x[7]);
        reinterpret_cast<uint4*>(args.jobs[j].y + row * kD)[chunk] = out;
      }
    }
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
  dim3 grid((T + kProTokens - 1) / kProTokens);
  {
    TraceScope trace_("prologue_kernel", stream);
    prologue_kernel<<<grid, 256, 0, stream>>>(args, turns, cu, S, T, eps, status_word());
  }
  return check_launch("prologue_kernel");
}

}  // namespace msa
