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
// rows' loads are issued before the angles are computed.  The kernel is bound
// by instruction issue as much as by memory, so the per-row work is kept
// short: a cursor (tensor, row) walks the thread's rows without a table
// lookup or a division per row, the token of a row is a multiply and a shift,
// and the arithmetic runs on packed pairs of fp32 (two channels per
// instruction).
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
constexpr int kProMaxH = 256;                // heads per tensor (token of a row = r * inv >> 20)
// forward kernel: 128 threads, 8 rows side by side with 16 threads per row
// (8 channels each: thread c < 8 holds the rotated pairs (4c + e, 4c + 32 + e),
// c >= 8 the pass-through channels 64 + 8 (c - 8) ..); four rows per thread in
// registers, so three rows' loads are in flight while the fourth is
// normalised, rotated and stored; the thread's weights stay in registers
// (66 registers, 7 CTAs per SM: a 16k pack's 1024 CTAs still run in one wave)
constexpr int kPfThreads = 128;
constexpr int kPfLanes = 16;
constexpr int kPfSlots = kPfThreads / kPfLanes;
static_assert(kPfThreads == kProTokens * (kRopeDim / 8), "one thread per (token, 4 frequencies)");

// the rows of one tensor that a CTA owns: rows [rowbase, rowbase + nrows) of
// its [T * H, 128] view, row r of them belonging to the CTA's token r / H
struct ProJobRows {
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  int nrows;        // ntok * H (0: tensor absent)
  int rowbase;      // t0 * H
  uint32_t inv;     // ceil(2^20 / H): r / H == (r * inv) >> 20 for r < 16 H, H <= 256
  int pad;
};

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
}

// (cos, sin) of one token's frequencies 4g .. 4g + 3 (thread = (token, g)):
// the token's position is found by a binary search over cu, the angle in
// turns by the 64-bit fixed-point product described above
__device__ __forceinline__ void rope_table_entry(float4 (*cs)[2][kRopeDim / 8], const RopeTurns& turns,
                                                 const int32_t* __restrict__ cu, int S, int T,
                                                 int t0, int tid) {
  const int qt = tid >> 3, g = tid & 7;
  const int t = t0 + qt;
  float cv[4] = {1.f, 1.f, 1.f, 1.f}, sv[4] = {0.f, 0.f, 0.f, 0.f};
  if (t < T) {
    int lo = 0, hi = S;   // largest s with cu[s] <= t
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
    }
    const unsigned long long pos = static_cast<unsigned long long>(t - __ldg(cu + lo));
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const long long ang = static_cast<long long>(pos * turns.f[4 * g + e]);
      sincospif(static_cast<float>(ang) * 1.0842021724855044e-19f, &sv[e], &cv[e]);   // * 2^-63
    }
  }
  cs[qt][0][g] = make_float4(cv[0], cv[1], cv[2], cv[3]);
  cs[qt][1][g] = make_float4(sv[0], sv[1], sv[2], sv[3]);
}

__global__ void __launch_bounds__(kPfThreads, 7) prologue_kernel(const PrologueArgs args,
                                                                  const RopeTurns turns,
                                                                  const int32_t* __restrict__ cu,
                                                                  int S, int T, float eps,
                                                                  uint32_t* status) {
  pdl_enter();
  __shared__ __align__(16) float4 cs[kProTokens][2][kRopeDim / 8];
  __shared__ __align__(16) float wsh[4][kD];
  __shared__ ProJobRows js[4];
  const int t0 = blockIdx.x * kProTokens;
  const int tid = threadIdx.x;
  const int ntok = min(kProTokens, T - t0);
  const int c = tid & (kPfLanes - 1);     // channel group of the row
  const int slot = tid / kPfLanes;
  // channel offsets (elements) of this thread's two 4-channel pieces
  const int off0 = (c < 8) ? 4 * c : 64 + 8 * (c - 8);
  const int off1 = (c < 8) ? 4 * c + 32 : 64 + 8 * (c - 8) + 4;
  if (tid < 4) {
    const int H = args.hstart[tid + 1] - args.hstart[tid];
    ProJobRows r;
    r.x = args.jobs[tid].x;
    r.y = args.jobs[tid].y;
    r.nrows = ntok * H;
    r.rowbase = t0 * H;
    r.inv = H > 0 ? ((1u << 20) + H - 1) / H : 0u;
    r.pad = 0;
    js[tid] = r;
  }
  __syncthreads();

  // The thread's rows are the CTA's rows slot, slot + 8, slot + 16, ... taken
  // tensor by tensor; the cursor (cj, cr) = (tensor, row within its CTA rows)
  // and that tensor's fields stay in registers between rows.
  int cj = 0, cr = slot, cnr = 0, crb = 0;
  uint32_t cinv = 0;
  const __nv_bfloat16* cx = nullptr;
  auto next_tensor = [&]() {
    while (cj < 4 && cr >= js[cj].nrows) {
      cr -= js[cj].nrows;
      ++cj;
    }
    if (cj < 4) {
      cx = js[cj].x;
      cnr = js[cj].nrows;
      crb = js[cj].rowbase;
      cinv = js[cj].inv;
    }
  };
  next_tensor();
  struct Rows {
    uint2 xa, xb;
    int g;     // row of the tensor's [T * H, 128] view
    int jt;    // tensor | token of the CTA << 2; -1: none
  };
  Rows ra, rb, rc, rd;
  auto load_row = [&](Rows& R) {
    R.jt = -1;
    R.g = 0;
    R.xa = make_uint2(0, 0);
    R.xb = R.xa;
    if (cj < 4) {
      const int g = crb + cr;
      const __nv_bfloat16* src = cx + static_cast<size_t>(g) * kD;
      R.xa = __ldcs(reinterpret_cast<const uint2*>(src + off0));
      R.xb = __ldcs(reinterpret_cast<const uint2*>(src + off1));
      R.g = g;
      R.jt = cj | static_cast<int>((static_cast<uint32_t>(cr) * cinv) >> 20) << 2;
      cr += kPfSlots;
      if (cr >= cnr) next_tensor();
    }
  };
  // the first rows' loads are in flight while the weights and angles are set up
  load_row(ra);
  load_row(rb);
  load_row(rc);
  for (int k = tid; k < 4 * kD; k += blockDim.x) {
    const int j = k / kD;
    wsh[j][k % kD] = (args.hstart[j] < args.hstart[j + 1])
                         ? 1.f + __bfloat162float(args.jobs[j].w[k % kD]) : 0.f;
  }
  rope_table_entry(cs, turns, cu, S, T, t0, tid);
  __syncthreads();

  // 1 + w of the thread's 8 channels for tensor wj, in registers; reloaded
  // when a row of another tensor comes up (three times per thread at most)
  int wj = -1;
  float2 w2[4];
  auto process = [&](const Rows& R) {
    const int j = R.jt < 0 ? 0 : (R.jt & 3);
    const int tl = R.jt < 0 ? 0 : (R.jt >> 2);
    if (j != wj) {
      const float4 w0 = *reinterpret_cast<const float4*>(&wsh[j][off0]);
      const float4 w1 = *reinterpret_cast<const float4*>(&wsh[j][off1]);
      w2[0] = make_float2(w0.x, w0.y);
      w2[1] = make_float2(w0.z, w0.w);
      w2[2] = make_float2(w1.x, w1.y);
      w2[3] = make_float2(w1.z, w1.w);
      wj = j;
    }
    // x: channels off0 + {0,1}, off0 + {2,3}, off1 + {0,1}, off1 + {2,3}
    float2 x[4] = {bf2_to_f2(R.xa.x), bf2_to_f2(R.xa.y), bf2_to_f2(R.xb.x), bf2_to_f2(R.xb.y)};
    float2 s2 = __fmul2_rn(x[0], x[0]);
#pragma unroll
    for (int e = 1; e < 4; ++e) s2 = __ffma2_rn(x[e], x[e], s2);
    float ss = s2.x + s2.y;
    // x (1 + w) while the sum of squares is reduced
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = __fmul2_rn(x[e], w2[e]);
#pragma unroll
    for (int m = kPfLanes / 2; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    if (c < 8) {
      // rotate channel 4c + e (x1) with 4c + 32 + e (x2), frequency 4c + e:
      // x1' = x1 cos - x2 sin, x2' = x2 cos + x1 sin (pairs e = 0,1 and 2,3)
      const float4 cv = cs[tl][0][c], sv = cs[tl][1][c];
      const float2 c2[2] = {make_float2(cv.x, cv.y), make_float2(cv.z, cv.w)};
      const float2 s2v[2] = {make_float2(sv.x, sv.y), make_float2(sv.z, sv.w)};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float2 x1 = x[h], x2 = x[2 + h];
        // x1 cos - x2 sin as x1 cos + (-x2) sin: the sign goes on the product's operand
        const float2 nx2 = make_float2(-x2.x, -x2.y);
        x[h] = __ffma2_rn(x1, c2[h], __fmul2_rn(nx2, s2v[h]));
        x[2 + h] = __ffma2_rn(x2, c2[h], __fmul2_rn(x1, s2v[h]));
      }
    }
    const float rinv = rsqrtf(ss * (1.f / kD) + eps);
    const float2 rr = make_float2(rinv, rinv);
    if (R.jt >= 0) {
      uint2 oa, ob;
      const float2 y0 = __fmul2_rn(x[0], rr), y1 = __fmul2_rn(x[1], rr);
      const float2 y2 = __fmul2_rn(x[2], rr), y3 = __fmul2_rn(x[3], rr);
      oa.x = pack_bf16x2(y0.x, y0.y);
      oa.y = pack_bf16x2(y1.x, y1.y);
      ob.x = pack_bf16x2(y2.x, y2.y);
      ob.y = pack_bf16x2(y3.x, y3.y);
      __nv_bfloat16* dst = js[j].y + static_cast<size_t>(R.g) * kD;
      *reinterpret_cast<uint2*>(dst + off0) = oa;
      *reinterpret_cast<uint2*>(dst + off1) = ob;
    }
  };
  // the loop bound is uniform over the CTA: every lane reaches the shuffles;
  // three rows' loads are in flight while the fourth row is processed
  const int rows = ntok * args.hstart[4];
  for (int base = 0; base < rows; base += 4 * kPfSlots) {
    load_row(rd);
    process(ra);
    if (base + kPfSlots >= rows) break;
    load_row(ra);
    process(rb);
    if (base + 2 * kPfSlots >= rows) break;
    load_row(rb);
    process(rc);
    if (base + 3 * kPfSlots >= rows) break;
    load_row(rc);
    process(rd);
  }
}

msa_status_t launch_prologue(const PrologueJob* jobs, int njobs, const int32_t* cu, int S, int T,
                             float rope_base, float eps, cudaStream_t stream) {
  if (njobs < 1 || njobs > 4) return fail(MSA_ERR_INVALID_ARG, "prologue takes 1..4 tensors");
  for (int j = 0; j < njobs; ++j)
    if (jobs[j].H > kProMaxH)
      return fail(MSA_ERR_UNSUPPORTED, "prologue: at most %d heads per tensor (got %d)", kProMaxH,
                  jobs[j].H);
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
// the third is processed.  Few live values per thread keep 7 CTAs on an SM;
// the thread's 8 weights stay in registers, the token of a row is a multiply
// and a shift, and the arithmetic runs on packed pairs of fp32.
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
  __shared__ __align__(16) float4 cs[kProTokens][2][kRopeDim / 8];
  __shared__ float red[kPbSlots][kD + 4];
  const int tid = threadIdx.x;
  const int c = tid & (kPbLanes - 1);
  const int slot = tid / kPbLanes;
  const int off0 = (c < 8) ? 4 * c : 64 + 8 * (c - 8);
  const int off1 = (c < 8) ? 4 * c + 32 : 64 + 8 * (c - 8) + 4;
  const uint32_t inv = ((1u << 20) + H - 1) / H;   // r / H == (r * inv) >> 20 (r < 16 H)
  // 1 + w of the thread's 8 channels, and their dw sums over its rows
  float2 w2[4];
  {
    const uint2 wa = __ldg(reinterpret_cast<const uint2*>(w + off0));
    const uint2 wb = __ldg(reinterpret_cast<const uint2*>(w + off1));
    const float2 one = make_float2(1.f, 1.f);
    w2[0] = __fadd2_rn(bf2_to_f2(wa.x), one);
    w2[1] = __fadd2_rn(bf2_to_f2(wa.y), one);
    w2[2] = __fadd2_rn(bf2_to_f2(wb.x), one);
    w2[3] = __fadd2_rn(bf2_to_f2(wb.y), one);
  }
  float2 aw[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) aw[e] = make_float2(0.f, 0.f);
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
    Rows ra, rb, rc;
    __syncthreads();                       // the previous group's angles are consumed
    load_rows(slot, ra);                   // in flight while the angles are computed
    load_rows(kPbSlots + slot, rb);
    rope_table_entry(cs, turns, cu, S, T, t0, tid);
    __syncthreads();

    auto process = [&](const Rows& R) {
      const bool valid = R.r >= 0;
      const int tl = valid ? static_cast<int>((static_cast<uint32_t>(R.r) * inv) >> 20) : 0;
      float2 xv[4] = {bf2_to_f2(R.xa.x), bf2_to_f2(R.xa.y), bf2_to_f2(R.xb.x), bf2_to_f2(R.xb.y)};
      float2 dz[4] = {bf2_to_f2(R.ga.x), bf2_to_f2(R.ga.y), bf2_to_f2(R.gb.x), bf2_to_f2(R.gb.y)};
      float2 s2 = __fmul2_rn(xv[0], xv[0]);
#pragma unroll
      for (int e = 1; e < 4; ++e) s2 = __ffma2_rn(xv[e], xv[e], s2);
      float ss = s2.x + s2.y;
#pragma unroll
      for (int m = kPbLanes / 2; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      if (c < 8) {
        // dz = R^T dy for the pairs (4c + e, 4c + 32 + e), frequency 4c + e:
        // d1' = d1 cos + d2 sin, d2' = d2 cos - d1 sin
        const float4 cv = cs[tl][0][c], sv = cs[tl][1][c];
        const float2 c2[2] = {make_float2(cv.x, cv.y), make_float2(cv.z, cv.w)};
        const float2 s2v[2] = {make_float2(sv.x, sv.y), make_float2(sv.z, sv.w)};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float2 d1 = dz[h], d2 = dz[2 + h];
          const float2 nd1 = make_float2(-d1.x, -d1.y);
          dz[h] = __ffma2_rn(d1, c2[h], __fmul2_rn(d2, s2v[h]));
          dz[2 + h] = __ffma2_rn(d2, c2[h], __fmul2_rn(nd1, s2v[h]));
        }
      }
      const float rinv = rsqrtf(ss * (1.f / kD) + eps);
      const float2 rr = make_float2(rinv, rinv);
      float2 gw[4];
      float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        xv[e] = __fmul2_rn(xv[e], rr);     // xh
        gw[e] = __fmul2_rn(dz[e], w2[e]);  // g = dz (1 + w)
        d2 = __ffma2_rn(gw[e], xv[e], d2);
      }
      float dot = d2.x + d2.y;
#pragma unroll
      for (int m = kPbLanes / 2; m >= 1; m >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, m);
      const float nmean = dot * (-1.f / kD);
      if (valid) {
        const float2 nm = make_float2(nmean, nmean);
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 v = __fmul2_rn(__ffma2_rn(xv[e], nm, gw[e]), rr);   // r (g - xh mean)
          o[e] = pack_bf16x2(v.x, v.y);
          aw[e] = __ffma2_rn(dz[e], xv[e], aw[e]);
        }
        __nv_bfloat16* dr = dx + (row_base + R.r) * kD;
        *reinterpret_cast<uint2*>(dr + off0) = make_uint2(o[0], o[1]);
        *reinterpret_cast<uint2*>(dr + off1) = make_uint2(o[2], o[3]);
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
  for (int e = 0; e < 2; ++e) {
    red[slot][off0 + 2 * e] = aw[e].x;
    red[slot][off0 + 2 * e + 1] = aw[e].y;
    red[slot][off1 + 2 * e] = aw[2 + e].x;
    red[slot][off1 + 2 * e + 1] = aw[2 + e].y;
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
  if (H > kProMaxH)
    return fail(MSA_ERR_UNSUPPORTED, "prologue backward: at most %d heads (got %d)", kProMaxH, H);
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
