// Fused prologue: per-head Gemma RMSNorm, x / sqrt(mean(x^2) + eps) * (1 + w),
// followed by partial RoPE on the first 64 of 128 channels (channel i pairs
// with i + 32; angle = position * base^(-2i/64)).  ("MiniMax-M3.1-Flash",
// 1 "Model Introduction"; "MiniMax-M3" Megatron-Bridge page, "Architecture
// Notes".)  bf16 [T, H, 128] -> bf16 [T, H, 128] (in place allowed); HBM-bound.
//
// Layout of the work: a CTA takes 8 consecutive tokens of one tensor.  Its 256
// threads first compute the 8 x 32 (cos, sin) pairs of those tokens once, then
// sweep the 8 x H rows, 16 threads per row, 8 channels (16 bytes) per thread.
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
  int ctas_per_job;      // ceil(T / 8)
};

constexpr int kProTokens = 8;

__global__ void __launch_bounds__(256) prologue_kernel(const PrologueArgs args,
                                                       const RopeTurns turns,
                                                       const int32_t* __restrict__ cu, int S,
                                                       int T, float eps, uint32_t* status) {
  __shared__ float2 cs[kProTokens][kRopeDim / 2];
  const int job_id = blockIdx.x / args.ctas_per_job;
  const int t0 = (blockIdx.x % args.ctas_per_job) * kProTokens;
  const PrologueJob job = args.jobs[job_id];
  const int tid = threadIdx.x;

  // (cos, sin) for the CTA's 8 tokens: thread = (token, frequency)
  {
    const int tl = tid >> 5, i = tid & 31;
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

  const int H = job.H;
  const int chunk = tid & 15;           // 8 channels: [8 chunk, 8 chunk + 8)
  float w[8];
  {
    const uint4 wv = __ldg(reinterpret_cast<const uint4*>(job.w) + chunk);
    const __nv_bfloat162* wp = reinterpret_cast<const __nv_bfloat162*>(&wv);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 f = __bfloat1622float2(wp[j]);
      w[2 * j] = 1.f + f.x;
      w[2 * j + 1] = 1.f + f.y;
    }
  }
  const int ntok = min(kProTokens, T - t0);
  const int rows = ntok * H;
  for (int r = tid >> 4; r < ((rows + 15) & ~15); r += 16) {
    const bool valid = r < rows;
    const int tl = valid ? r / H : 0;
    const size_t row = static_cast<size_t>(t0) * H + (valid ? r : 0);
    const uint4* src = reinterpret_cast<const uint4*>(job.x + row * kD) + chunk;
    uint4* dst = reinterpret_cast<uint4*>(job.y + row * kD) + chunk;
    float x[8];
    uint4 xv = valid ? *src : make_uint4(0, 0, 0, 0);
    {
      const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&xv);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 f = __bfloat1622float2(xp[j]);
        x[2 * j] = f.x;
        x[2 * j + 1] = f.y;
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(x[j], x[j], ss);
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const float rinv = rsqrtf(ss * (1.f / kD) + eps);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = x[j] * rinv * w[j];
    // rotate-half on channels [0, 64): chunk c < 4 holds x1, chunk c + 4 holds x2
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = __shfl_xor_sync(0xffffffffu, x[j], 4);
    if (chunk < 8) {
      const int fbase = (chunk & 3) * 8;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 c = cs[tl][fbase + j];
        x[j] = (chunk < 4) ? (x[j] * c.x - y[j] * c.y) : (x[j] * c.x + y[j] * c.y);
      }
    }
    if (valid) {
      uint4 out;
      out.x = pack_bf16x2(x[0], x[1]);
      out.y = pack_bf16x2(x[2], x[3]);
      out.z = pack_bf16x2(x[4], x[5]);
      out.w = pack_bf16x2(x[6], x[7]);
      *dst = out;
    }
  }
}

msa_status_t launch_prologue(const PrologueJob* jobs, int njobs, const int32_t* cu, int S, int T,
                             float rope_base, float eps, cudaStream_t stream) {
  PrologueArgs args{};
  for (int j = 0; j < njobs; ++j) args.jobs[j] = jobs[j];
  args.ctas_per_job = (T + kProTokens - 1) / kProTokens;
  RopeTurns turns;
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < kRopeDim / 2; ++i) {
    double f = std::pow(static_cast<double>(rope_base), -2.0 * i / kRopeDim);
    turns.f[i] = static_cast<unsigned long long>(f / two_pi * 18446744073709551616.0);
  }
  dim3 grid(args.ctas_per_job * njobs);
  {
    TraceScope trace_("prologue_kernel", stream);
    prologue_kernel<<<grid, 256, 0, stream>>>(args, turns, cu, S, T, eps, status_word());
  }
  return check_launch("prologue_kernel");
}

}  // namespace msa
