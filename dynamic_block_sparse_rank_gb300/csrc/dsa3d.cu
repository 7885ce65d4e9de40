// 3D deformable sliding attention: the offset network and the sampled-window
// attention ("MegaSlide-DiT", gist.science explainer, section 2 "3D deformable
// sliding attention (3D-DSA)": keys and values sampled by trilinear
// interpolation in a kt x kh x kw neighbourhood moved by offsets that a light
// 3D convolution and a linear layer predict; linear cost in N).
//
// Neither step is a dense contraction worth the tensor cores: the offset
// network is a 27-tap depthwise convolution and a d x 3S matrix per token
// (3S = 81 outputs for a 3x3x3 window), and the attention is a batch of
// per-token gathers of 8 S key and value rows with no operand shared between
// tokens.  Both are SIMT kernels whose bound is the gather traffic through L1
// (the rows of a token's neighbourhood are re-read by its neighbours) and the
// FP32 pipe; HBM sees each input row about once.
//
//   dsa3d_offsets_kernel  64 raster tokens x one head per CTA.  Stage 1: a
//                         thread owns a channel pair and runs the 27-tap
//                         depthwise convolution for 16 or 8 tokens (zero
//                         padding), into shared memory as [channel][token].
//                         Stage 2: the d x 3S matrix, staged in shared memory
//                         96 columns at a time, is applied as a register-tiled
//                         product (4 tokens x 6 outputs per thread, packed
//                         fp32x2 FMAs).
//   dsa3d_fwd_kernel      a warp serves 256/d tokens of one head, a token's
//                         row split over d/8 lanes (16 bytes each); per
//                         window point the 8 trilinear corners
//                         inside the raster are gathered (K and V rows, one
//                         contiguous 128- or 256-byte row per corner), the logit
//                         is the corner-weighted q.k reduced across the
//                         token's lanes, and an online softmax (base 2)
//                         accumulates the corner-weighted v (packed fp32x2
//                         FMAs).  Positions are tested against the
//                         raster in float before any index is formed, so a
//                         non-finite offset only moves its sample outside.
//
// Backward (the loss reaching the attention through O):
//   dsa3d_bwd_kernel      the forward's warp layout; one gather of the corners
//                         per window point gives P_s, dP_s, k~_s and the
//                         corner weights' derivatives, from which dq and the
//                         offsets' gradient follow (both linear in D); each
//                         sample's coefficients are stored and the sample is
//                         counted in the cell of its floor position.
//   dsa3d_cell_scan_kernel, dsa3d_cell_fill_kernel
//                         bucket the samples by cell (exclusive scan of the
//                         counts, then one record per sample in its cell).
//   dsa3d_dkdv_kernel     each dK / dV row gathered from the records of the 8
//                         cells it is a corner of: rows written once, no
//                         atomics.
//   dsa3d_offsets_bwd_kernel, dsa3d_offsets_bwd_conv_kernel
//                         the offset network: dY, dWl, dbl per token tile,
//                         then the transposed convolution into dQ with dWc
//                         and dbc.
#include <cuda_bf16.h>

#include "internal.h"

namespace sda {

namespace {

constexpr int kDsaTok = 32;     // tokens per CTA, both kernels
constexpr int kDsaThreads = 256;

__device__ __forceinline__ void raster_coords(int n, int H, int W, int& t, int& y, int& x) {
  x = n % W;
  const int r = n / W;
  y = r % H;
  t = r / H;
}

constexpr int kOffTok = 64;     // tokens per CTA of the offset network
constexpr int kOffJ = 96;       // outputs per pass: 16 groups of 6
constexpr int kOffYStride = kOffTok + 4;  // floats per channel row of Y (float4-aligned)

__host__ __device__ constexpr size_t offsets_smem_bytes(int D) {
  return (size_t)D * kOffYStride * 4 + (size_t)D * kOffJ * 4;
}

// Y[c][tok] = bc + sum over the 27 taps of Wc * Q (zero outside the raster) for the kOffTok
// raster tokens from n0 of head h, into Ys ([D][kOffYStride], all 256 threads).  A thread owns a
// channel pair: its 54 taps stay in registers, its loads are 4-byte pieces of one 128- or
// 256-byte row per warp, kPer tokens' loads in flight together.  Tokens at or past N get bc.
template <int D, int kPer>
__device__ __forceinline__ void conv_tile(const __nv_bfloat16* __restrict__ Q, const float* __restrict__ Wc,
                                          const float* __restrict__ bc, const Dsa3dArgs& a, int b, int h, int n0,
                                          float* Ys) {
  constexpr int kPairs = D / 2;
  constexpr int kGroups = kDsaThreads / kPairs;
  static_assert((kOffTok / kGroups) % kPer == 0, "tokens per thread must divide by kPer");
  const int N = a.T * a.H * a.W;
  const int tid = threadIdx.x;
  const int cp = tid % kPairs, tg = tid / kPairs;
  const int c0 = 2 * cp;
  float w0[27], w1[27];
  const float* wc0 = Wc + ((long long)h * D + c0) * 27;
#pragma unroll
  for (int k = 0; k < 27; ++k) {
    w0[k] = wc0[k];
    w1[k] = wc0[27 + k];
  }
  const float b0 = bc[h * D + c0], b1 = bc[h * D + c0 + 1];
  const __nv_bfloat16* Qh = Q + (long long)b * N * a.heads * D + (long long)h * D + c0;
  for (int tok = tg; tok < kOffTok; tok += kPer * kGroups) {
    uint32_t v[kPer][27];
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int n = n0 + tok + e * kGroups;
      int t = 0, y = 0, x = 0;
      if (n < N) raster_coords(n, a.H, a.W, t, y, x);
#pragma unroll
      for (int k = 0; k < 27; ++k) {
        const int tt = t + k / 9 - 1, yy = y + (k / 3) % 3 - 1, xx = x + k % 3 - 1;
        const bool in = n < N && tt >= 0 && tt < a.T && yy >= 0 && yy < a.H && xx >= 0 && xx < a.W;
        const int m = (tt * a.H + yy) * a.W + xx;
        v[e][k] = in ? __ldg(reinterpret_cast<const unsigned*>(Qh + (long long)m * a.heads * D)) : 0u;
      }
    }
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      float y0 = b0, y1 = b1;
#pragma unroll
      for (int k = 0; k < 27; ++k) {
        const float2 f = bf16x2_to_f2(v[e][k]);  // zero bits outside the raster: zero padding
        y0 = fmaf(w0[k], f.x, y0);
        y1 = fmaf(w1[k], f.y, y1);
      }
      Ys[c0 * kOffYStride + tok + e * kGroups] = y0;
      Ys[(c0 + 1) * kOffYStride + tok + e * kGroups] = y1;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kDsaThreads) dsa3d_offsets_kernel(const __nv_bfloat16* __restrict__ Q,
                                                                   const float* __restrict__ Wc,
                                                                   const float* __restrict__ bc,
                                                                   const float* __restrict__ Wl,
                                                                   const float* __restrict__ bl,
                                                                   float* __restrict__ off, Dsa3dArgs a) {
  extern __shared__ __align__(16) float dsmem[];
  float* Ys = dsmem;                      // [D][kOffYStride]
  float* Ws = dsmem + D * kOffYStride;   // [D][kOffJ]: one pass's columns of Wl[h]
  const int h = blockIdx.y, b = blockIdx.z;
  const int N = a.T * a.H * a.W;
  const int n0 = blockIdx.x * kOffTok;
  const int tid = threadIdx.x;

  // Stage 1: Y[c][tok] = bc + sum over the 27 taps of Wc * Q (zero outside the raster).
  conv_tile<D, 2>(Q, Wc, bc, a, b, h, n0, Ys);

  // Stage 2: off[tok][j] = bl[j] + sum_c Y[c][tok] Wl[h][c][j].  Register tiles of 4 tokens x 6
  // outputs per thread (16 x 16 threads cover 64 tokens x 96 outputs per pass).
  const int S3 = 3 * a.S;
  const int tg = tid / 16, jg = tid % 16;
  const float* wl = Wl + (long long)h * D * S3;
  for (int j0 = 0; j0 < S3; j0 += kOffJ) {
    __syncthreads();  // Y written (first pass) / the previous pass's Ws read
    for (int e = tid; e < D * kOffJ; e += kDsaThreads) {
      const int c = e / kOffJ, jj = e % kOffJ;
      Ws[e] = j0 + jj < S3 ? wl[(long long)c * S3 + j0 + jj] : 0.f;
    }
    __syncthreads();
    float2 acc[4][3];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const int j = j0 + jg * 6 + 2 * q;
        acc[i][q] = make_float2(j < S3 ? bl[h * S3 + j] : 0.f, j + 1 < S3 ? bl[h * S3 + j + 1] : 0.f);
      }
#pragma unroll 4
    for (int c = 0; c < D; ++c) {
      const float4 y4 = *reinterpret_cast<const float4*>(Ys + c * kOffYStride + tg * 4);
      const float2* wr = reinterpret_cast<const float2*>(Ws + c * kOffJ + jg * 6);
      const float2 wv[3] = {wr[0], wr[1], wr[2]};
      const float yv[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 3; ++q) acc[i][q] = ffma2(make_float2(yv[i], yv[i]), wv[q], acc[i][q]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = n0 + tg * 4 + i;
      if (n >= N) continue;
      float* orow = off + (((long long)b * N + n) * a.heads + h) * S3;
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const int j = j0 + jg * 6 + 2 * q;
        if (j < S3) orow[j] = acc[i][q].x;
        if (j + 1 < S3) orow[j + 1] = acc[i][q].y;
      }
    }
  }
}

// Dot product of 8 bf16 pairs (4 packed words each): .x sums the low halves, .y the high
// ones.  A mixed-precision FMA takes the bf16 operands as they are (their product is exact
// in fp32) and adds it to the fp32 sum with one rounding, so neither row is unpacked.
__device__ __forceinline__ float2 dot8_bf16(const uint32_t (&a)[4], const uint32_t (&b)[4]) {
  float lo = 0.f, hi = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\tfma.rn.f32.bf16 %1, ah, bh, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(a[i]), "r"(b[i]));
  return make_float2(lo, hi);
}

// A warp serves 256 / D tokens of one head: a token's row is split over D / 8 lanes, 8
// channels (16 bytes) each.  Per window point the three axes give the two candidate grid
// coordinates, their weights (1 - f, f) and whether each lies inside the raster; the 8
// corners combine them, and only corners inside with a non-zero weight are gathered.
template <int D>
__global__ void __launch_bounds__(kDsaThreads) dsa3d_fwd_kernel(const __nv_bfloat16* __restrict__ Q,
                                                               const __nv_bfloat16* __restrict__ K,
                                                               const __nv_bfloat16* __restrict__ V,
                                                               const float* __restrict__ off,
                                                               __nv_bfloat16* __restrict__ O, float* __restrict__ LSE,
                                                               Dsa3dArgs a) {
  constexpr int LPT = D / 8;       // lanes per token
  constexpr int TPW = 32 / LPT;    // tokens per warp at a time
  constexpr int kWarps = kDsaThreads / 32;
  constexpr int kPerWarp = kDsaTok / kWarps;  // tokens per warp
  constexpr float kLog2e = 1.4426950408889634f;
  const int h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = lane / LPT, sl = lane % LPT;
  const int N = a.T * a.H * a.W;
  const long long rs = (long long)a.heads * D;  // elements between consecutive tokens' rows
  const __nv_bfloat16* Kb = K + (long long)b * N * rs + (long long)h * D + sl * 8;
  const __nv_bfloat16* Vb = V + (long long)b * N * rs + (long long)h * D + sl * 8;
  const int rt = (a.kt - 1) / 2, rh = (a.kh - 1) / 2, rw = (a.kw - 1) / 2;
  const float Tm = (float)(a.T - 1), Hm = (float)(a.H - 1), Wm = (float)(a.W - 1);
  const int HW = a.H * a.W;
  for (int u = 0; u < kPerWarp; u += TPW) {
    const int n_raw = blockIdx.x * kDsaTok + warp * kPerWarp + u + slot;
    const bool valid = n_raw < N;
    const int n = valid ? n_raw : N - 1;  // lanes of a missing token compute a copy and store nothing
    int t, y, x;
    raster_coords(n, a.H, a.W, t, y, x);
    const long long row = ((long long)b * N + n) * rs + (long long)h * D + sl * 8;
    // q stays in bf16: q . k is formed with mixed-precision FMAs (bf16 x bf16 products are
    // exact in fp32), and the scale (to base-2 logits) is applied to the reduced sum.
    const float qs = a.scale * kLog2e;
    uint32_t q[4];
    {
      const uint4 qv = __ldg(reinterpret_cast<const uint4*>(Q + row));
      q[0] = qv.x, q[1] = qv.y, q[2] = qv.z, q[3] = qv.w;
    }
    const float* offn = off + (((long long)b * N + n) * a.heads + h) * (3LL * a.S);
    float m = -INFINITY, l = 0.f;
    float2 o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = make_float2(0.f, 0.f);
    // offsets of the current window point; the next point's are loaded one point ahead,
    // so their latency overlaps this point's gathers
    float ox = __ldg(offn), oy = __ldg(offn + 1), oz = __ldg(offn + 2);
    int s = 0;
    for (int wa = 0; wa < a.kt; ++wa)
      for (int wb = 0; wb < a.kh; ++wb)
        for (int wc = 0; wc < a.kw; ++wc, ++s) {
          const float pt = (float)(t + wa - rt) + ox;
          const float ph = (float)(y + wb - rh) + oy;
          const float pw = (float)(x + wc - rw) + oz;
          {
            const int sn = s + 1 < a.S ? s + 1 : s;
            ox = __ldg(offn + 3 * sn), oy = __ldg(offn + 3 * sn + 1), oz = __ldg(offn + 3 * sn + 2);
          }
          const float bt = floorf(pt), bh = floorf(ph), bw = floorf(pw);
          const float ft = pt - bt, fh = ph - bh, fw = pw - bw;
          // per axis: is coordinate base (+1) inside the raster; tested in float, so NaN or
          // far-out positions fail here and form no index
          const bool t0 = bt >= 0.f && bt <= Tm, t1 = bt >= -1.f && bt <= Tm - 1.f;
          const bool h0 = bh >= 0.f && bh <= Hm, h1 = bh >= -1.f && bh <= Hm - 1.f;
          const bool w0 = bw >= 0.f && bw <= Wm, w1 = bw >= -1.f && bw <= Wm - 1.f;
          const float wt[2] = {1.f - ft, ft}, wh[2] = {1.f - fh, fh}, ww[2] = {1.f - fw, fw};
          const bool vt[2] = {t0, t1}, vh[2] = {h0, h1}, vw[2] = {w0, w1};
          // base index from coordinates clamped to [-1, max]: only corners found inside use it
          const int it = (int)fminf(fmaxf(bt, -1.f), Tm), ih = (int)fminf(fmaxf(bh, -1.f), Hm),
                    iw = (int)fminf(fmaxf(bw, -1.f), Wm);
          const int m000 = (it * a.H + ih) * a.W + iw;
          float dot = 0.f;
          float2 vs[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) vs[i] = make_float2(0.f, 0.f);
#pragma unroll
          for (int corner = 0; corner < 8; ++corner) {
            const int ct = corner >> 2, ch = (corner >> 1) & 1, cw = corner & 1;
            const float wgt = wt[ct] * wh[ch] * ww[cw];
            if (!(vt[ct] && vh[ch] && vw[cw]) || wgt == 0.f) continue;
            const long long mrow = (long long)(m000 + ct * HW + ch * a.W + cw) * rs;
            const uint4 kv = __ldg(reinterpret_cast<const uint4*>(Kb + mrow));
            const uint4 vv = __ldg(reinterpret_cast<const uint4*>(Vb + mrow));
            const uint32_t kw4[4] = {kv.x, kv.y, kv.z, kv.w}, vw4[4] = {vv.x, vv.y, vv.z, vv.w};
            const float2 pd = dot8_bf16(q, kw4);
            const float2 w2 = make_float2(wgt, wgt);
#pragma unroll
            for (int i = 0; i < 4; ++i) vs[i] = ffma2(w2, bf16x2_to_f2(vw4[i]), vs[i]);
            dot = fmaf(wgt, pd.x + pd.y, dot);
          }
#pragma unroll
          for (int sh = LPT / 2; sh > 0; sh >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, sh);
          dot *= qs;
          const float mn = fmaxf(m, dot);
          const float corr = exp2f(m - mn), p = exp2f(dot - mn);
          l = fmaf(l, corr, p);
          const float2 c2 = make_float2(corr, corr), p2 = make_float2(p, p);
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = ffma2(o[i], c2, make_float2(p2.x * vs[i].x, p2.y * vs[i].y));
          m = mn;
        }
    if (valid) {
      const float inv = 1.f / l;
      uint32_t w4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 r = __floats2bfloat162_rn(o[i].x * inv, o[i].y * inv);
        w4[i] = *reinterpret_cast<uint32_t*>(&r);
      }
      *reinterpret_cast<uint4*>(O + row) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      if (sl == 0) LSE[((long long)b * a.heads + h) * N + n] = (m + log2f(l)) * 0.6931471805599453f;
    }
  }
}

// Floor cell, fractional position and per-axis inside flags of a sample position (token units).
// Every test is in float: a NaN position fails them all, and no index is formed from it.
struct SampleCell {
  float f[3];
  bool v0[3], v1[3];  // the lower / upper corner on that axis is inside the raster
  int ib[3];          // the floor, clamped to -1 .. size - 1
  int cell;           // index among cell_entries(), -1 when no corner is inside
};

// Cells of one (batch entry, head): the (T+1) x (H+1) x (W+1) floor positions -1 .. T-1 etc.,
// plus one entry for the total.
__host__ __device__ inline long long cell_entries(const Dsa3dArgs& a) {
  return (long long)(a.T + 1) * (a.H + 1) * (a.W + 1) + 1;
}

__device__ __forceinline__ SampleCell sample_cell(const float (&pc)[3], const Dsa3dArgs& a) {
  SampleCell c;
  const float mx[3] = {(float)(a.T - 1), (float)(a.H - 1), (float)(a.W - 1)};
#pragma unroll
  for (int ax = 0; ax < 3; ++ax) {
    const float bse = floorf(pc[ax]);
    c.f[ax] = pc[ax] - bse;
    c.v0[ax] = bse >= 0.f && bse <= mx[ax];
    c.v1[ax] = bse >= -1.f && bse <= mx[ax] - 1.f;
    c.ib[ax] = (int)fminf(fmaxf(bse, -1.f), mx[ax]);
  }
  const bool any = (c.v0[0] || c.v1[0]) && (c.v0[1] || c.v1[1]) && (c.v0[2] || c.v1[2]);
  c.cell = any ? ((c.ib[0] + 1) * (a.H + 1) + c.ib[1] + 1) * (a.W + 1) + c.ib[2] + 1 : -1;
  return c;
}

// Backward of the window attention (dLSE = 0), per token, in one gather of the corners.  The
// same warp layout as the forward.  For every window point the corners' K and V rows give the
// logit q.k~_s (so P_s = exp(a_s - LSE), the forward's LSE), dP_s = dO.v~_s, k~_s itself, and
// the weights' derivatives applied to q.K_c and dO.V_c per axis (GK_s, GV_s).  Everything that
// needs D = sum_s P_s dP_s is linear in it: with da_s = P_s (dP_s - D),
//   dq = scale sum_s da_s k~_s = scale (sum_s P_s dP_s k~_s - D sum_s P_s k~_s)
// (two register accumulators), and the offset gradient scale da_s GK_s + P_s GV_s is formed
// after the loop from (P_s, dP_s, GK_s, GV_s) kept in shared memory, one sample per lane.  dK
// and dV are not scattered from here: every sample's coefficients (scale da_s, P_s) go to
// `coef`, and the sample is counted in the cell of the grid that holds its floor position
// (cells -1 .. T-1 per axis, so that every cell with a corner inside the raster has one), for
// dsa3d_dkdv_kernel to gather.
constexpr int kSampleWords = 9;  // P, dP, GK[3], GV[3], cell

// token slots of a CTA (8 warps x 256 / D tokens side by side) x S samples x kSampleWords
__host__ __device__ constexpr size_t bwd_smem_bytes(int D, int S) {
  return (size_t)(kDsaThreads / 32) * (256 / D) * S * kSampleWords * 4;
}

// Sums 8 values over the LPT lanes of a token group by halving: after it lane sl holds the
// total of value sl / (LPT / 8) (8 shuffles for LPT = 16, 7 for LPT = 8, instead of 8 full
// reductions).
template <int LPT>
__device__ __forceinline__ float reduce8(const float (&v)[8], int sl) {
  const bool hA = sl & (LPT / 2), hB = sl & (LPT / 4), hC = sl & (LPT / 8);
  float a[4], b2[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = hA ? v[i] : v[i + 4], keep = hA ? v[i + 4] : v[i];
    a[i] = keep + __shfl_xor_sync(0xffffffffu, send, LPT / 2);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = hB ? a[i] : a[i + 2], keep = hB ? a[i + 2] : a[i];
    b2[i] = keep + __shfl_xor_sync(0xffffffffu, send, LPT / 4);
  }
  float c = (hC ? b2[1] : b2[0]) + __shfl_xor_sync(0xffffffffu, hC ? b2[0] : b2[1], LPT / 8);
#pragma unroll
  for (int o = LPT / 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  return c;
}

template <int D>
__global__ void __launch_bounds__(kDsaThreads, 3) dsa3d_bwd_kernel(const __nv_bfloat16* __restrict__ Q,
                                                               const __nv_bfloat16* __restrict__ K,
                                                               const __nv_bfloat16* __restrict__ V,
                                                               const float* __restrict__ off,
                                                               const float* __restrict__ LSE,
                                                               const __nv_bfloat16* __restrict__ dO,
                                                               float* __restrict__ dQ, float2* __restrict__ coef,
                                                               int* __restrict__ count, float* __restrict__ doff,
                                                               Dsa3dArgs a) {
  constexpr int LPT = D / 8;
  constexpr int TPW = 32 / LPT;
  constexpr int kWarps = kDsaThreads / 32;
  constexpr int kPerWarp = kDsaTok / kWarps;
  constexpr int kSub = LPT / 8;  // lanes holding the same reduced value
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ float bsm[];  // [kWarps * TPW token slots][S][kSampleWords]
  const int h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = lane / LPT, sl = lane % LPT;
  const int N = a.T * a.H * a.W;
  const long long rs = (long long)a.heads * D;
  const long long hb = (long long)b * N * rs + (long long)h * D + sl * 8;  // this head's lane offset, batch b
  const int rt = (a.kt - 1) / 2, rh = (a.kh - 1) / 2, rw = (a.kw - 1) / 2;
  const int HW = a.H * a.W;
  float* rec = bsm + (size_t)(warp * TPW + slot) * a.S * kSampleWords;
  auto load8 = [&](const __nv_bfloat16* p, float2 (&v)[4]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    v[0] = bf16x2_to_f2(u.x);
    v[1] = bf16x2_to_f2(u.y);
    v[2] = bf16x2_to_f2(u.z);
    v[3] = bf16x2_to_f2(u.w);
  };
  for (int u = 0; u < kPerWarp; u += TPW) {
    const int n_raw = blockIdx.x * kDsaTok + warp * kPerWarp + u + slot;
    const bool valid = n_raw < N;
    const int n = valid ? n_raw : N - 1;  // lanes of a missing token compute a copy and write nothing
    int t, y, x;
    raster_coords(n, a.H, a.W, t, y, x);
    float2 q[4];
    load8(Q + hb + (long long)n * rs, q);
    uint32_t g[4];  // dO stays in bf16: dO . V takes mixed-precision FMAs (dot8_bf16)
    {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(dO + hb + (long long)n * rs));
      g[0] = u.x, g[1] = u.y, g[2] = u.z, g[3] = u.w;
    }
    const float lse2 = LSE[((long long)b * a.heads + h) * N + n] * kLog2e;
    const float sl2 = a.scale * kLog2e;
    const long long ns = ((long long)b * N + n) * a.heads + h;
    const float* offn = off + ns * (3LL * a.S);
    float2 acc_pd[4], acc_p[4];  // sum_s P_s dP_s k~_s, sum_s P_s k~_s (this lane's 8 channels)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc_pd[i] = acc_p[i] = make_float2(0.f, 0.f);
    float Dsum = 0.f;
    int s = 0;
    for (int wa = 0; wa < a.kt; ++wa)
      for (int wb = 0; wb < a.kh; ++wb)
        for (int wc = 0; wc < a.kw; ++wc, ++s) {
          const float pc[3] = {(float)(t + wa - rt) + __ldg(offn + 3 * s),
                               (float)(y + wb - rh) + __ldg(offn + 3 * s + 1),
                               (float)(x + wc - rw) + __ldg(offn + 3 * s + 2)};
          const SampleCell c = sample_cell(pc, a);
          const int m000 = (c.ib[0] * a.H + c.ib[1]) * a.W + c.ib[2];
          float2 ks[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) ks[i] = make_float2(0.f, 0.f);
          // partial sums over this lane's channels: w q.K, w dO.V, then dw/dpos q.K and dw/dpos dO.V per axis
          float v8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int corner = 0; corner < 8; ++corner) {
            const int ct = corner >> 2, ch = (corner >> 1) & 1, cw = corner & 1;
            const bool in = (ct ? c.v1[0] : c.v0[0]) && (ch ? c.v1[1] : c.v0[1]) && (cw ? c.v1[2] : c.v0[2]);
            if (!in) continue;
            const float wt = ct ? c.f[0] : 1.f - c.f[0], wh = ch ? c.f[1] : 1.f - c.f[1],
                        ww = cw ? c.f[2] : 1.f - c.f[2];
            const float w = wt * wh * ww;
            const long long row = (long long)(m000 + ct * HW + ch * a.W + cw) * rs;
            float2 kv[4];
            load8(K + hb + row, kv);
            const uint4 vu = __ldg(reinterpret_cast<const uint4*>(V + hb + row));
            const uint32_t vv[4] = {vu.x, vu.y, vu.z, vu.w};
            float2 pq = make_float2(0.f, 0.f);
            const float2 pv = dot8_bf16(g, vv);
            const float2 w2 = make_float2(w, w);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              pq = ffma2(q[i], kv[i], pq);
              ks[i] = ffma2(w2, kv[i], ks[i]);
            }
            const float pqs = pq.x + pq.y, pvs = pv.x + pv.y;
            const float dt = (ct ? 1.f : -1.f) * wh * ww, dh = (ch ? 1.f : -1.f) * wt * ww,
                        dw = (cw ? 1.f : -1.f) * wt * wh;
            v8[0] = fmaf(w, pqs, v8[0]);
            v8[1] = fmaf(w, pvs, v8[1]);
            v8[2] = fmaf(dt, pqs, v8[2]);
            v8[3] = fmaf(dh, pqs, v8[3]);
            v8[4] = fmaf(dw, pqs, v8[4]);
            v8[5] = fmaf(dt, pvs, v8[5]);
            v8[6] = fmaf(dh, pvs, v8[6]);
            v8[7] = fmaf(dw, pvs, v8[7]);
          }
          const float r = reduce8<LPT>(v8, sl);  // total of value sl / kSub
          const float logit = __shfl_sync(0xffffffffu, r, slot * LPT);
          const float dP = __shfl_sync(0xffffffffu, r, slot * LPT + kSub);
          const float Ps = exp2f(fmaf(logit, sl2, -lse2));
          const float pd = Ps * dP;
          Dsum += pd;
          const float2 pd2 = make_float2(pd, pd), p2 = make_float2(Ps, Ps);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc_pd[i] = ffma2(pd2, ks[i], acc_pd[i]);
            acc_p[i] = ffma2(p2, ks[i], acc_p[i]);
          }
          if (sl % kSub == 0) {
            const int k = sl / kSub;
            float* rs9 = rec + s * kSampleWords;
            rs9[k] = k == 0 ? Ps : r;  // P, dP, GK[3], GV[3]
            if (k == 0) rs9[8] = __int_as_float(c.cell);
          }
        }
    __syncwarp();
    if (valid) {
      float4 o[2];
      float* of = reinterpret_cast<float*>(o);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        of[2 * i] = a.scale * fmaf(-Dsum, acc_p[i].x, acc_pd[i].x);
        of[2 * i + 1] = a.scale * fmaf(-Dsum, acc_p[i].y, acc_pd[i].y);
      }
      float4* dqr = reinterpret_cast<float4*>(dQ + hb + (long long)n * rs);
      dqr[0] = o[0];
      dqr[1] = o[1];
      // per sample, one lane each: the offset gradient, the coefficients, the cell count
      for (int s2 = sl; s2 < a.S; s2 += LPT) {
        const float* rs9 = rec + s2 * kSampleWords;
        const float Ps = rs9[0], sda = a.scale * Ps * (rs9[1] - Dsum);
        float* od = doff + ns * (3LL * a.S) + 3 * s2;
        od[0] = fmaf(sda, rs9[2], Ps * rs9[5]);
        od[1] = fmaf(sda, rs9[3], Ps * rs9[6]);
        od[2] = fmaf(sda, rs9[4], Ps * rs9[7]);
        coef[ns * a.S + s2] = make_float2(sda, Ps);
        const int cell = __float_as_int(rs9[8]);
        if (cell >= 0) atomicAdd(count + ((long long)b * a.heads + h) * cell_entries(a) + cell, 1);
      }
    }
    __syncwarp();  // the records are rewritten by the next token
  }
}

// ---- dK and dV of the window attention, gathered per row: the samples counted per cell by
// dsa3d_bwd_kernel are bucketed by cell (an exclusive scan of the counts, then a fill), and a
// row m = (t, y, x) sums the contributions of the samples in the 8 cells (t, y, x) - {0, 1}^3,
// whose corner it is: dK[m] = sum w scale da q_n, dV[m] = sum w P dO_n, w the sample's
// trilinear weight at m.  Every row is written once, by one thread group: no atomics on rows.

// Exclusive prefix sum of one (batch entry, head)'s cell counts, in place: count[e] becomes the
// first record of cell e (count[E] the total), copied to cursor for the fill.  One CTA per
// (batch entry, head); a round stages 8,192 entries in shared memory with coalesced loads,
// each thread scans 8 consecutive ones (skewed rows: no bank conflicts), and the round is
// stored back coalesced.
constexpr int kScanPer = 8;
constexpr int kScanRound = 1024 * kScanPer;

__device__ __forceinline__ int scan_skew(int i) { return i + (i >> 5); }

__global__ void __launch_bounds__(1024) dsa3d_cell_scan_kernel(int* __restrict__ count, int* __restrict__ cursor,
                                                               long long ncell) {
  __shared__ int buf[kScanRound + kScanRound / 32];
  __shared__ int wsum[32];
  int* c = count + blockIdx.x * ncell;
  int* cur = cursor + blockIdx.x * ncell;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int carry = 0;
  for (long long base = 0; base < ncell; base += kScanRound) {
#pragma unroll
    for (int k = 0; k < kScanPer; ++k) {
      const int i = k * 1024 + tid;
      buf[scan_skew(i)] = base + i < ncell ? c[base + i] : 0;
    }
    __syncthreads();
    int v[kScanPer];
    int tsum = 0;
#pragma unroll
    for (int k = 0; k < kScanPer; ++k) {
      v[k] = buf[scan_skew(kScanPer * tid + k)];
      tsum += v[k];
    }
    int x = tsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      wsum[lane] = w;
    }
    __syncthreads();
    int e = carry + (warp ? wsum[warp - 1] : 0) + x - tsum;
#pragma unroll
    for (int k = 0; k < kScanPer; ++k) {
      buf[scan_skew(kScanPer * tid + k)] = e;
      e += v[k];
    }
    carry += wsum[31];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kScanPer; ++k) {
      const int i = k * 1024 + tid;
      if (base + i < ncell) {
        const int o = buf[scan_skew(i)];
        c[base + i] = o;
        cur[base + i] = o;
      }
    }
    __syncthreads();  // buf and wsum are rewritten next round
  }
}

// One thread per (token, window point): the sample's floor cell and fractional position,
// computed as dsa3d_bwd_kernel computes them (sample_cell), and its record written at the next
// free place of its cell: (token, f_t, f_h, f_w) and (scale da, P).
__global__ void __launch_bounds__(kDsaThreads) dsa3d_cell_fill_kernel(const float* __restrict__ off,
                                                                     const float2* __restrict__ coef,
                                                                     int* __restrict__ cursor,
                                                                     int4* __restrict__ rec,
                                                                     float2* __restrict__ rcoef, Dsa3dArgs a) {
  const int h = blockIdx.y, b = blockIdx.z;
  const int N = a.T * a.H * a.W;
  const long long NS = (long long)N * a.S;
  const long long idx = (long long)blockIdx.x * kDsaThreads + threadIdx.x;
  if (idx >= NS) return;
  const int n = (int)(idx / a.S), s = (int)(idx % a.S);
  int t, y, x;
  raster_coords(n, a.H, a.W, t, y, x);
  const int wa = s / (a.kh * a.kw), wb = (s / a.kw) % a.kh, wc = s % a.kw;
  const long long ns = ((long long)b * N + n) * a.heads + h;
  const float* o = off + ns * (3LL * a.S) + 3 * s;
  const float pc[3] = {(float)(t + wa - (a.kt - 1) / 2) + __ldg(o), (float)(y + wb - (a.kh - 1) / 2) + __ldg(o + 1),
                       (float)(x + wc - (a.kw - 1) / 2) + __ldg(o + 2)};
  const SampleCell c = sample_cell(pc, a);
  if (c.cell < 0) return;
  const long long bh = (long long)b * a.heads + h;
  const int slot = atomicAdd(cursor + bh * cell_entries(a) + c.cell, 1);
  if (slot >= NS) return;  // only if this count disagreed with dsa3d_bwd_kernel's: never write past the records
  rec[bh * NS + slot] = make_int4(n, __float_as_int(c.f[0]), __float_as_int(c.f[1]), __float_as_int(c.f[2]));
  rcoef[bh * NS + slot] = __ldg(coef + ns * a.S + s);
}

// dK, dV rows gathered from the bucketed records, in the forward's warp layout (a row split
// over D / 8 lanes of 16 bytes, 256 / D rows per warp side by side).
template <int D>
__global__ void __launch_bounds__(kDsaThreads) dsa3d_dkdv_kernel(const __nv_bfloat16* __restrict__ Q,
                                                                const __nv_bfloat16* __restrict__ dO,
                                                                const int* __restrict__ start,
                                                                const int4* __restrict__ rec,
                                                                const float2* __restrict__ rcoef,
                                                                float* __restrict__ dK, float* __restrict__ dV,
                                                                Dsa3dArgs a) {
  constexpr int LPT = D / 8;
  constexpr int TPW = 32 / LPT;
  constexpr int kWarps = kDsaThreads / 32;
  constexpr int kPerWarp = kDsaTok / kWarps;
  const int h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = lane / LPT, sl = lane % LPT;
  const int N = a.T * a.H * a.W;
  const long long rs = (long long)a.heads * D;
  const long long hb = (long long)b * N * rs + (long long)h * D + sl * 8;
  const long long bh = (long long)b * a.heads + h;
  const int* st = start + bh * cell_entries(a);
  const int4* rc = rec + bh * ((long long)N * a.S);
  const float2* cf = rcoef + bh * ((long long)N * a.S);
  for (int u = 0; u < kPerWarp; u += TPW) {
    const int m = blockIdx.x * kDsaTok + warp * kPerWarp + u + slot;
    if (m >= N) continue;  // no shuffles below: a group may leave alone
    int t, y, x;
    raster_coords(m, a.H, a.W, t, y, x);
    float2 ak[4], av[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) ak[i] = av[i] = make_float2(0.f, 0.f);
#pragma unroll 1
    for (int corner = 0; corner < 8; ++corner) {
      const int ct = corner >> 2, ch = (corner >> 1) & 1, cw = corner & 1;
      const int cell = ((t - ct + 1) * (a.H + 1) + y - ch + 1) * (a.W + 1) + x - cw + 1;
      const int i1 = __ldg(st + cell + 1);
      for (int i = __ldg(st + cell); i < i1; ++i) {
        const int4 r = __ldg(rc + i);
        const float2 c = __ldg(cf + i);
        const float f0 = __int_as_float(r.y), f1 = __int_as_float(r.z), f2 = __int_as_float(r.w);
        const float w = (ct ? f0 : 1.f - f0) * (ch ? f1 : 1.f - f1) * (cw ? f2 : 1.f - f2);
        const uint4 qu = __ldg(reinterpret_cast<const uint4*>(Q + hb + (long long)r.x * rs));
        const uint4 gu = __ldg(reinterpret_cast<const uint4*>(dO + hb + (long long)r.x * rs));
        const float2 wk = make_float2(w * c.x, w * c.x), wv = make_float2(w * c.y, w * c.y);
        ak[0] = ffma2(wk, bf16x2_to_f2(qu.x), ak[0]);
        ak[1] = ffma2(wk, bf16x2_to_f2(qu.y), ak[1]);
        ak[2] = ffma2(wk, bf16x2_to_f2(qu.z), ak[2]);
        ak[3] = ffma2(wk, bf16x2_to_f2(qu.w), ak[3]);
        av[0] = ffma2(wv, bf16x2_to_f2(gu.x), av[0]);
        av[1] = ffma2(wv, bf16x2_to_f2(gu.y), av[1]);
        av[2] = ffma2(wv, bf16x2_to_f2(gu.z), av[2]);
        av[3] = ffma2(wv, bf16x2_to_f2(gu.w), av[3]);
      }
    }
    float* dkr = dK + hb + (long long)m * rs;
    float* dvr = dV + hb + (long long)m * rs;
    reinterpret_cast<float4*>(dkr)[0] = make_float4(ak[0].x, ak[0].y, ak[1].x, ak[1].y);
    reinterpret_cast<float4*>(dkr)[1] = make_float4(ak[2].x, ak[2].y, ak[3].x, ak[3].y);
    reinterpret_cast<float4*>(dvr)[0] = make_float4(av[0].x, av[0].y, av[1].x, av[1].y);
    reinterpret_cast<float4*>(dvr)[1] = make_float4(av[2].x, av[2].y, av[3].x, av[3].y);
  }
}

// Offset network backward, part 1 (gradients of the linear layer): for 64-token tiles of one
// (batch entry, head), with G = the tile's d_offsets, dY = G Wl[h]^T goes to the workspace
// ([B, N, heads, D] fp32), dWl[h] += Y^T G and dbl[h] += the column sums of G, Y recomputed
// by conv_tile.  The 3S outputs go in passes of 96 columns; a pass walks all of the CTA's
// tiles (every gridDim.x-th), adds its share of dY into the workspace (the first pass writes
// it; one thread owns an element in every pass) and keeps its dWl / dbl columns in registers
// until the pass ends, then adds them into dWl / dbl with atomics.  A 3 x 3 x 3 window takes
// one pass; each further pass recomputes Y.
constexpr int kGStride = kOffJ + 4;  // floats per token row of the staged d_offsets columns

__host__ __device__ constexpr int wlt_stride(int D) { return D + 4; }

__host__ __device__ constexpr size_t offsets_bwd_smem_bytes(int D) {
  return ((size_t)D * kOffYStride + (size_t)kOffTok * kGStride + (size_t)kOffJ * wlt_stride(D)) * 4;
}

template <int D>
__global__ void __launch_bounds__(kDsaThreads, 1)
    dsa3d_offsets_bwd_kernel(const __nv_bfloat16* __restrict__ Q, const float* __restrict__ Wc,
                             const float* __restrict__ bc, const float* __restrict__ Wl,
                             const float* __restrict__ doff, float* __restrict__ dY, float* __restrict__ dWl,
                             float* __restrict__ dbl, Dsa3dArgs a) {
  constexpr int CPT = D / 16;  // channels per thread in both register tiles
  extern __shared__ __align__(16) float dsmem[];
  float* Ys = dsmem;                     // [D][kOffYStride]
  float* Gs = Ys + D * kOffYStride;      // [kOffTok][kGStride]: one pass's d_offsets columns
  float* WlT = Gs + kOffTok * kGStride;  // [kOffJ][D + 4]: the same columns of Wl[h], transposed
  const int h = blockIdx.y, b = blockIdx.z;
  const int N = a.T * a.H * a.W;
  const int S3 = 3 * a.S;
  const int ntiles = (N + kOffTok - 1) / kOffTok;
  const int tid = threadIdx.x;
  const float* wl = Wl + (long long)h * D * S3;
  // dY tile: channels c1 .. c1 + CPT - 1 x tokens 4 tg1 .. 4 tg1 + 3
  const int c1 = (tid % 16) * CPT, tg1 = tid / 16;
  // dWl tile: channels cg2 + 16 k (k < CPT; interleaved, so the two channel groups of a warp
  // read different banks of Ys) x columns 6 jg2 .. 6 jg2 + 5 of the pass
  const int jg2 = tid % 16, cg2 = tid / 16;

  for (int j0 = 0; j0 < S3; j0 += kOffJ) {
    const int jn = min(kOffJ, S3 - j0);
    __syncthreads();  // the previous pass's WlT reads are done
    for (int e = tid; e < D * kOffJ; e += kDsaThreads) {
      const int c = e / kOffJ, jj = e % kOffJ;
      WlT[jj * wlt_stride(D) + c] = jj < jn ? wl[(long long)c * S3 + j0 + jj] : 0.f;
    }
    float2 gw[CPT][3];  // dWl[h][cg2 + 16 k][j0 + 6 jg2 + 2 q, + 1]
    float2 gb[3];       // dbl[h][the same columns]
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      gb[q] = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < CPT; ++k) gw[k][q] = make_float2(0.f, 0.f);
    }
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const int n0 = tile * kOffTok;
      __syncthreads();  // the previous tile's Ys / Gs reads are done
      conv_tile<D, 1>(Q, Wc, bc, a, b, h, n0, Ys);
      static_assert((kOffTok * kOffJ) % kDsaThreads == 0, "G staging must tile evenly");
#pragma unroll 8
      for (int e = tid; e < kOffTok * kOffJ; e += kDsaThreads) {
        const int tok = e / kOffJ, jj = e % kOffJ;
        const int n = n0 + tok;
        // rows past N and columns past 3S stay zero: they add nothing to dY, dWl or dbl
        Gs[tok * kGStride + jj] =
            n < N && jj < jn ? __ldg(doff + (((long long)b * N + n) * a.heads + h) * S3 + j0 + jj) : 0.f;
      }
      __syncthreads();

      // dY[tok][c] (+)= sum_j G[tok][j] Wl[h][c][j] over this pass's columns
      float2 acc[CPT][2];  // tokens (4 tg1, 4 tg1 + 1) and (4 tg1 + 2, 4 tg1 + 3)
#pragma unroll
      for (int k = 0; k < CPT; ++k) acc[k][0] = acc[k][1] = make_float2(0.f, 0.f);
#pragma unroll 4
      for (int jj = 0; jj < jn; ++jj) {
        const float* gcol = Gs + (4 * tg1) * kGStride + jj;
        const float2 g01 = make_float2(gcol[0], gcol[kGStride]);
        const float2 g23 = make_float2(gcol[2 * kGStride], gcol[3 * kGStride]);
        float w[CPT];
#pragma unroll
        for (int k = 0; k < CPT; k += 4) {
          const float4 w4 = *reinterpret_cast<const float4*>(WlT + jj * wlt_stride(D) + c1 + k);
          w[k] = w4.x;
          w[k + 1] = w4.y;
          w[k + 2] = w4.z;
          w[k + 3] = w4.w;
        }
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
          acc[k][0] = ffma2(make_float2(w[k], w[k]), g01, acc[k][0]);
          acc[k][1] = ffma2(make_float2(w[k], w[k]), g23, acc[k][1]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = n0 + 4 * tg1 + i;
        if (n >= N) continue;
        float* row = dY + (((long long)b * N + n) * a.heads + h) * D + c1;
#pragma unroll
        for (int k = 0; k < CPT; k += 4) {
          float4 v;
          v.x = (i & 1) ? acc[k][i >> 1].y : acc[k][i >> 1].x;
          v.y = (i & 1) ? acc[k + 1][i >> 1].y : acc[k + 1][i >> 1].x;
          v.z = (i & 1) ? acc[k + 2][i >> 1].y : acc[k + 2][i >> 1].x;
          v.w = (i & 1) ? acc[k + 3][i >> 1].y : acc[k + 3][i >> 1].x;
          float4* p = reinterpret_cast<float4*>(row + k);
          if (j0 > 0) {
            const float4 o = *p;
            v.x += o.x;
            v.y += o.y;
            v.z += o.z;
            v.w += o.w;
          }
          *p = v;
        }
      }

      // dWl[h][c][j] += sum_tok Y[c][tok] G[tok][j]; dbl[h][j] += sum_tok G[tok][j]
#pragma unroll 2
      for (int tok = 0; tok < kOffTok; ++tok) {
        const float2* grow = reinterpret_cast<const float2*>(Gs + tok * kGStride + 6 * jg2);
        const float2 g[3] = {grow[0], grow[1], grow[2]};
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
          const float y = Ys[(cg2 + 16 * k) * kOffYStride + tok];
#pragma unroll
          for (int q = 0; q < 3; ++q) gw[k][q] = ffma2(make_float2(y, y), g[q], gw[k][q]);
        }
#pragma unroll
        for (int q = 0; q < 3; ++q) gb[q] = fadd2(gb[q], g[q]);
      }
    }
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int j = j0 + 6 * jg2 + 2 * q;
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        float* p = dWl + ((long long)h * D + cg2 + 16 * k) * S3 + j;
        if (j < S3) atomicAdd(p, gw[k][q].x);
        if (j + 1 < S3) atomicAdd(p + 1, gw[k][q].y);
      }
      if (cg2 == 0) {
        if (j < S3) atomicAdd(dbl + (long long)h * S3 + j, gb[q].x);
        if (j + 1 < S3) atomicAdd(dbl + (long long)h * S3 + j + 1, gb[q].y);
      }
    }
  }
}

// Offset network backward, part 2 (gradients of the depthwise convolution): with dY from part
// 1, dQ[m][c] += sum over taps of Wc[h][c][tap] dY[m - tap][c] (the transposed convolution,
// zero padding), dWc[h][c][tap] += sum_m dY[m - tap][c] Q[m][c] and dbc[h][c] += sum_m dY[m][c].
// A thread owns one channel (the warp reads one 128-byte piece of a row per tap) and 256 / D
// tokens run side by side, two per thread at a time; the CTA walks 32-token tiles with the
// grid's x stride, keeps its 27 + 1 weight-gradient sums in registers and adds them with
// atomics at the end.
constexpr int kConvTok = 32;

template <int D>
__global__ void __launch_bounds__(kDsaThreads, 2)
    dsa3d_offsets_bwd_conv_kernel(const __nv_bfloat16* __restrict__ Q, const float* __restrict__ Wc,
                                  const float* __restrict__ dY, float* __restrict__ dQ, float* __restrict__ dWc,
                                  float* __restrict__ dbc, Dsa3dArgs a) {
  constexpr int kLanes = kDsaThreads / D;
  static_assert(kConvTok % (2 * kLanes) == 0, "two tokens per thread per step");
  const int h = blockIdx.y, b = blockIdx.z;
  const int N = a.T * a.H * a.W;
  const int ntiles = (N + kConvTok - 1) / kConvTok;
  const int c = threadIdx.x % D, lane = threadIdx.x / D;
  const long long rs = (long long)a.heads * D;  // elements between consecutive tokens' rows
  const long long base = (long long)b * N * rs + (long long)h * D + c;
  float w[27], gw[27];
#pragma unroll
  for (int k = 0; k < 27; ++k) {
    w[k] = Wc[((long long)h * D + c) * 27 + k];
    gw[k] = 0.f;
  }
  float gb = 0.f;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    for (int tok = lane; tok < kConvTok; tok += 2 * kLanes) {
      float v[2][27];
      float q[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int m = tile * kConvTok + tok + e * kLanes;
        int t = 0, y = 0, x = 0;
        if (m < N) raster_coords(m, a.H, a.W, t, y, x);
        q[e] = m < N ? __bfloat162float(Q[base + (long long)m * rs]) : 0.f;
#pragma unroll
        for (int k = 0; k < 27; ++k) {
          // tap k reads X at (t, y, x) + (k / 9, k / 3 % 3, k % 3) - 1 for the output at n = m - that
          const int tt = t - k / 9 + 1, yy = y - (k / 3) % 3 + 1, xx = x - k % 3 + 1;
          const bool in = m < N && tt >= 0 && tt < a.T && yy >= 0 && yy < a.H && xx >= 0 && xx < a.W;
          const int n = (tt * a.H + yy) * a.W + xx;
          v[e][k] = in ? __ldg(dY + base + (long long)n * rs) : 0.f;
        }
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int m = tile * kConvTok + tok + e * kLanes;
        float dq = 0.f;
#pragma unroll
        for (int k = 0; k < 27; ++k) {
          dq = fmaf(w[k], v[e][k], dq);
          gw[k] = fmaf(v[e][k], q[e], gw[k]);
        }
        gb += v[e][13];  // the centre tap: dY of the token itself
        if (m < N) dQ[base + (long long)m * rs] += dq;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 27; ++k) atomicAdd(dWc + ((long long)h * D + c) * 27 + k, gw[k]);
  atomicAdd(dbc + (long long)h * D + c, gb);
}

template <int D>
cudaError_t launch_dsa3d(const Dsa3dArgs& a, const __nv_bfloat16* Q, const __nv_bfloat16* K, const __nv_bfloat16* V,
                         const float* Wc, const float* bc, const float* Wl, const float* bl, float* off,
                         __nv_bfloat16* O, float* LSE, bool offsets, cudaStream_t st) {
  const long long N = (long long)a.T * a.H * a.W;
  if (offsets) {
    const size_t smem = offsets_smem_bytes(D);
    cudaError_t e =
        cudaFuncSetAttribute(dsa3d_offsets_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((N + kOffTok - 1) / kOffTok), a.heads, a.B);
    dsa3d_offsets_kernel<D><<<grid, kDsaThreads, smem, st>>>(Q, Wc, bc, Wl, bl, off, a);
  } else {
    const dim3 grid((unsigned)((N + kDsaTok - 1) / kDsaTok), a.heads, a.B);
    dsa3d_fwd_kernel<D><<<grid, kDsaThreads, 0, st>>>(Q, K, V, off, O, LSE, a);
  }
  note_launches(1);
  return cudaGetLastError();
}

// Workspace of the window attention's backward: per (batch entry, head) the samples'
// coefficients in token order, their records and coefficients in cell order, the cell starts
// and the fill cursors; 256-byte aligned pieces.
struct BwdWs {
  float2* coef;
  int4* rec;
  float2* rcoef;
  int* count;
  int* cursor;
  size_t count_bytes, bytes;
};

BwdWs bwd_ws_layout(const Dsa3dArgs& a, void* base) {
  const size_t samples = (size_t)a.B * a.heads * a.T * a.H * a.W * a.S;
  const size_t cells = (size_t)a.B * a.heads * cell_entries(a);
  size_t at = 0;
  auto take = [&](size_t bytes) {
    const size_t o = at;
    at = (at + bytes + 255) & ~(size_t)255;
    return o;
  };
  const size_t o_coef = take(samples * sizeof(float2)), o_rec = take(samples * sizeof(int4)),
               o_rcoef = take(samples * sizeof(float2)), o_count = take(cells * sizeof(int)),
               o_cursor = take(cells * sizeof(int));
  BwdWs w{};
  if (char* p = static_cast<char*>(base)) {
    w.coef = reinterpret_cast<float2*>(p + o_coef);
    w.rec = reinterpret_cast<int4*>(p + o_rec);
    w.rcoef = reinterpret_cast<float2*>(p + o_rcoef);
    w.count = reinterpret_cast<int*>(p + o_count);
    w.cursor = reinterpret_cast<int*>(p + o_cursor);
  }
  w.count_bytes = cells * sizeof(int);
  w.bytes = at;
  return w;
}

template <int D>
cudaError_t launch_dsa3d_bwd(const Dsa3dArgs& a, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                             const __nv_bfloat16* V, const float* off, const float* LSE, const __nv_bfloat16* dO,
                             float* dQ, float* dK, float* dV, float* doff, void* ws, cudaStream_t st) {
  const long long N = (long long)a.T * a.H * a.W;
  const BwdWs w = bwd_ws_layout(a, ws);
  cudaError_t e;
  if ((e = cudaMemsetAsync(w.count, 0, w.count_bytes, st)) != cudaSuccess) return e;
  const dim3 grid((unsigned)((N + kDsaTok - 1) / kDsaTok), a.heads, a.B);
  const size_t smem = bwd_smem_bytes(D, a.S);
  if ((e = cudaFuncSetAttribute(dsa3d_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
      cudaSuccess)
    return e;
  dsa3d_bwd_kernel<D><<<grid, kDsaThreads, smem, st>>>(Q, K, V, off, LSE, dO, dQ, w.coef, w.count, doff, a);
  dsa3d_cell_scan_kernel<<<a.B * a.heads, 1024, 0, st>>>(w.count, w.cursor, cell_entries(a));
  const dim3 fgrid((unsigned)((N * a.S + kDsaThreads - 1) / kDsaThreads), a.heads, a.B);
  dsa3d_cell_fill_kernel<<<fgrid, kDsaThreads, 0, st>>>(off, w.coef, w.cursor, w.rec, w.rcoef, a);
  dsa3d_dkdv_kernel<D><<<grid, kDsaThreads, 0, st>>>(Q, dO, w.count, w.rec, w.rcoef, dK, dV, a);
  note_launches(4);
  return cudaGetLastError();
}

// Persistent grid of part 1 / part 2 of the offset network backward: per (batch entry, head)
// as many CTAs as the device holds at once (capped by the tiles), so that the CTAs of one head
// run together and its rows' neighbours meet in L2.
template <typename K>
cudaError_t resident_ctas(K kernel, size_t smem, int tiles, int& ctas) {
  int dev = 0, sms = 0, occ = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kDsaThreads, smem)) != cudaSuccess) return e;
  ctas = max(1, min(tiles, max(1, occ) * sms));
  return cudaSuccess;
}

template <int D>
cudaError_t launch_dsa3d_offsets_bwd(const Dsa3dArgs& a, const __nv_bfloat16* Q, const float* Wc, const float* bc,
                                     const float* Wl, const float* doff, float* dQ, float* dWc, float* dbc,
                                     float* dWl, float* dbl, float* dY, cudaStream_t st) {
  const int N = a.T * a.H * a.W;
  const int S3 = 3 * a.S;
  cudaError_t e;
  // weight gradients are accumulated by atomics
  if ((e = cudaMemsetAsync(dWc, 0, (size_t)a.heads * D * 27 * sizeof(float), st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dbc, 0, (size_t)a.heads * D * sizeof(float), st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dWl, 0, (size_t)a.heads * D * S3 * sizeof(float), st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dbl, 0, (size_t)a.heads * S3 * sizeof(float), st)) != cudaSuccess) return e;
  const size_t smem = offsets_bwd_smem_bytes(D);
  if ((e = cudaFuncSetAttribute(dsa3d_offsets_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem)) != cudaSuccess)
    return e;
  int c1 = 0, c2 = 0;
  if ((e = resident_ctas(dsa3d_offsets_bwd_kernel<D>, smem, (N + kOffTok - 1) / kOffTok, c1)) != cudaSuccess)
    return e;
  if ((e = resident_ctas(dsa3d_offsets_bwd_conv_kernel<D>, 0, (N + kConvTok - 1) / kConvTok, c2)) != cudaSuccess)
    return e;
  dsa3d_offsets_bwd_kernel<D><<<dim3(c1, a.heads, a.B), kDsaThreads, smem, st>>>(Q, Wc, bc, Wl, doff, dY, dWl,
                                                                                  dbl, a);
  dsa3d_offsets_bwd_conv_kernel<D><<<dim3(c2, a.heads, a.B), kDsaThreads, 0, st>>>(Q, Wc, dY, dQ, dWc, dbc, a);
  note_launches(2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t dsa3d_bwd(const Dsa3dArgs& a, const void* Q, const void* K, const void* V, const float* off,
                      const float* LSE, const void* dO, float* dQ, float* dK, float* dV, float* doff, void* ws,
                      cudaStream_t st) {
  const auto* q = static_cast<const __nv_bfloat16*>(Q);
  const auto* k = static_cast<const __nv_bfloat16*>(K);
  const auto* v = static_cast<const __nv_bfloat16*>(V);
  const auto* g = static_cast<const __nv_bfloat16*>(dO);
  return a.d == 64 ? launch_dsa3d_bwd<64>(a, q, k, v, off, LSE, g, dQ, dK, dV, doff, ws, st)
                   : launch_dsa3d_bwd<128>(a, q, k, v, off, LSE, g, dQ, dK, dV, doff, ws, st);
}

size_t dsa3d_bwd_ws_bytes(const Dsa3dArgs& a) { return bwd_ws_layout(a, nullptr).bytes; }

cudaError_t dsa3d_offsets(const Dsa3dArgs& a, const void* Q, const float* Wc, const float* bc, const float* Wl,
                          const float* bl, float* off, cudaStream_t st) {
  const auto* q = static_cast<const __nv_bfloat16*>(Q);
  return a.d == 64 ? launch_dsa3d<64>(a, q, nullptr, nullptr, Wc, bc, Wl, bl, off, nullptr, nullptr, true, st)
                   : launch_dsa3d<128>(a, q, nullptr, nullptr, Wc, bc, Wl, bl, off, nullptr, nullptr, true, st);
}

cudaError_t dsa3d_fwd(const Dsa3dArgs& a, const void* Q, const void* K, const void* V, const float* off, void* O,
                      float* LSE, cudaStream_t st) {
  const auto* q = static_cast<const __nv_bfloat16*>(Q);
  const auto* k = static_cast<const __nv_bfloat16*>(K);
  const auto* v = static_cast<const __nv_bfloat16*>(V);
  auto* o = static_cast<__nv_bfloat16*>(O);
  return a.d == 64
             ? launch_dsa3d<64>(a, q, k, v, nullptr, nullptr, nullptr, nullptr, const_cast<float*>(off), o, LSE, false, st)
             : launch_dsa3d<128>(a, q, k, v, nullptr, nullptr, nullptr, nullptr, const_cast<float*>(off), o, LSE, false,
                                 st);
}

cudaError_t dsa3d_offsets_bwd(const Dsa3dArgs& a, const void* Q, const float* Wc, const float* bc, const float* Wl,
                              const float* doff, float* dQ, float* dWc, float* dbc, float* dWl, float* dbl,
                              void* ws, cudaStream_t st) {
  const auto* q = static_cast<const __nv_bfloat16*>(Q);
  auto* dY = static_cast<float*>(ws);
  return a.d == 64 ? launch_dsa3d_offsets_bwd<64>(a, q, Wc, bc, Wl, doff, dQ, dWc, dbc, dWl, dbl, dY, st)
                   : launch_dsa3d_offsets_bwd<128>(a, q, Wc, bc, Wl, doff, dQ, dWc, dbc, dWl, dbl, dY, st);
}

size_t dsa3d_offsets_bwd_ws_bytes(const Dsa3dArgs& a) {
  return (size_t)a.B * a.T * a.H * a.W * a.heads * a.d * sizeof(float);
}

}  // namespace sda
