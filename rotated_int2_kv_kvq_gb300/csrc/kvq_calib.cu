// kvq_calib.cu — OptR rotation calibration on the GPU (off the decode path).
//
// Method: "Output-Aware Rotation for INT2 KV-Cache Quantization" (pith.science
// review of arXiv 2608.02691).  Per KV head a correction of a base rotation,
// R = R0 exp(S) with S = A - A^T ("What carries the argument", mechanism (1)),
// is learned with Adam ("Assumptions & free parameters": 80 steps, lambda_K = 1)
// through the whole quantised path with a straight-through estimator for the
// rounding (mechanism (3)): first for keys, minimising KL(p || p~) plus lambda_K
// times the key-induced post-W_O error with values unquantised; then for values,
// minimising the value-induced post-W_O error with the quantised-key attention
// fixed (the error decomposition of "What carries the argument" and the referee
// report's Eqs. (14), (16)).  The objective is taken over the last Nq query
// positions of a causal calibration chunk.
//
// Structure: every contraction is one launch of a batched fp32 GEMM (batch =
// KV head); the quantiser, its straight-through backward, the causal softmax
// with its KL and backward, the post-W_O error and Adam are row or element
// kernels; exp(S) is scaling and squaring of a Taylor polynomial (carrying
// exp - I through the squarings), and the
// gradient with respect to S is the adjoint of the Frechet derivative of exp,
// L_exp(S^T, G), read from the upper-right block of exp([[S^T, G], [0, S^T]]).
// The host needs each step's largest |S| to pick the number of squarings, so a
// calibration call synchronises its stream once per objective evaluation (the
// adjoint's exponential reuses the forward one's norm).
#include <math.h>

#include <algorithm>
#include <cstdint>
#include <initializer_list>
#include <utility>
#include <vector>

#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kD = kDim;

// ---------------------------------------------------------------------------
// Batched fp32 GEMM: C[b] = alpha * op(A[b]) * op(B[b]) + beta * C[b], row-major.
// op(A) is M x K: A[m * lda + k], or, transposed, A stored K x M: A[k * lda + m].
// op(B) is K x N: B[k * ldb + n], or, transposed, B stored N x K: B[n * ldb + k].
// Two kernels: gemm_tile_kernel<BM, BK> (BM x BM tile, BK-deep k-slices (64
// for the 32-wide tile, 32 for the 64-wide one) double-buffered in shared
// memory with the next slice's 16-byte loads in flight while the current one
// is multiplied, 4 x 4 outputs per thread) when M and N are multiples of 32, K
// of 64, and every row starts on 16 bytes;
// otherwise gemm_kernel (64 x 64 tile, scalar guarded loads).  beta == 0 does
// not read C; diag adds diag * I (square C, ksplit 1).  With ksplit > 1 the K
// range is cut into ksplit chunks (blockIdx.z = batch * ksplit + chunk) whose
// partial products are added to C atomically (C zeroed beforehand when
// beta == 0).
// ---------------------------------------------------------------------------
struct Gemm {
  const float* A;
  const float* B;
  float* C;
  int M, N, K, lda, ldb, ldc;
  long long sA, sB, sC;
  float alpha, beta;
  int ta, tb;
  int ksplit, kchunk;
  float diag;
};

__global__ void __launch_bounds__(256) gemm_kernel(Gemm g) {
  __shared__ float As[16][68];
  __shared__ float Bs[16][68];
  const int bz = blockIdx.z / g.ksplit, kz = blockIdx.z % g.ksplit;
  const int kbeg = kz * g.kchunk, kend = min(g.K, kbeg + g.kchunk);
  const float* A = g.A + bz * g.sA;
  const float* B = g.B + bz * g.sB;
  float* C = g.C + bz * g.sC;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int k0 = kbeg; k0 < kend; k0 += 16) {
    for (int i = tid; i < 1024; i += 256) {
      int mm, kk;
      if (g.ta) { kk = i >> 6; mm = i & 63; } else { mm = i >> 4; kk = i & 15; }
      const int gm = m0 + mm, gk = k0 + kk;
      float v = 0.0f;
      if (gm < g.M && gk < kend)
        v = g.ta ? A[static_cast<long long>(gk) * g.lda + gm] : A[static_cast<long long>(gm) * g.lda + gk];
      As[kk][mm] = v;
    }
    for (int i = tid; i < 1024; i += 256) {
      int nn, kk;
      if (g.tb) { nn = i >> 4; kk = i & 15; } else { kk = i >> 6; nn = i & 63; }
      const int gn = n0 + nn, gk = k0 + kk;
      float v = 0.0f;
      if (gn < g.N && gk < kend)
        v = g.tb ? B[static_cast<long long>(gn) * g.ldb + gk] : B[static_cast<long long>(gk) * g.ldb + gn];
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 16 * j;
      if (n >= g.N) continue;
      float* c = C + static_cast<long long>(m) * g.ldc + n;
      if (g.ksplit > 1)
        atomicAdd(c, g.alpha * acc[i][j]);
      else
        *c = (g.beta == 0.0f ? g.alpha * acc[i][j] : fmaf(g.alpha, acc[i][j], g.beta * *c)) +
             (m == n ? g.diag : 0.0f);
    }
  }
}

template <int BM, int BK>
__global__ void __launch_bounds__((BM / 4) * (BM / 4)) gemm_tile_kernel(Gemm g) {
  constexpr int TPR = BM / 4, NT = TPR * TPR, KQ = BK / 4;
  constexpr int PER = BM * BK / 4 / NT;          // 16-byte loads per operand slice per thread
  __shared__ __align__(16) float As[2][BK][BM + 4];
  __shared__ __align__(16) float Bs[2][BK][BM + 4];
  const int bz = blockIdx.z / g.ksplit, kz = blockIdx.z % g.ksplit;
  const int kbeg = kz * g.kchunk, kend = min(g.K, kbeg + g.kchunk);
  const float* A = g.A + bz * g.sA;
  const float* B = g.B + bz * g.sB;
  float* C = g.C + bz * g.sC;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BM;
  const int tid = threadIdx.x, tx = tid % TPR, ty = tid / TPR;
  float4 ra[PER], rb[PER];
  auto load = [&](int k0) {
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int f = tid + p * NT;
      if (g.ta) {        // A stored K x M: rows of M
        const int kk = f / TPR, mm = 4 * (f % TPR);
        ra[p] = *reinterpret_cast<const float4*>(A + static_cast<long long>(k0 + kk) * g.lda + m0 + mm);
      } else {           // A stored M x K: rows of K
        const int mm = f / KQ, kk = 4 * (f % KQ);
        ra[p] = *reinterpret_cast<const float4*>(A + static_cast<long long>(m0 + mm) * g.lda + k0 + kk);
      }
      if (g.tb) {        // B stored N x K
        const int nn = f / KQ, kk = 4 * (f % KQ);
        rb[p] = *reinterpret_cast<const float4*>(B + static_cast<long long>(n0 + nn) * g.ldb + k0 + kk);
      } else {           // B stored K x N
        const int kk = f / TPR, nn = 4 * (f % TPR);
        rb[p] = *reinterpret_cast<const float4*>(B + static_cast<long long>(k0 + kk) * g.ldb + n0 + nn);
      }
    }
  };
  // Shared-memory column of element m in k-row kk: 4-element groups are
  // XOR-swizzled by (kk / 4) mod 8, so the transposing scalar stores of 4
  // consecutive k from 8 (or 16) rows spread over all banks while each group
  // stays one aligned 16-byte read.
  const auto col = [](int kk, int m) { return m ^ (((kk >> 2) & 7) << 2); };
  auto store = [&](int buf) {
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int f = tid + p * NT;
      if (g.ta) {
        const int kk = f / TPR, mm = 4 * (f % TPR);
        *reinterpret_cast<float4*>(&As[buf][kk][col(kk, mm)]) = ra[p];
      } else {
        const int mm = f / KQ, kk = 4 * (f % KQ);
        As[buf][kk][col(kk, mm)] = ra[p].x;
        As[buf][kk + 1][col(kk + 1, mm)] = ra[p].y;
        As[buf][kk + 2][col(kk + 2, mm)] = ra[p].z;
        As[buf][kk + 3][col(kk + 3, mm)] = ra[p].w;
      }
      if (g.tb) {
        const int nn = f / KQ, kk = 4 * (f % KQ);
        Bs[buf][kk][col(kk, nn)] = rb[p].x;
        Bs[buf][kk + 1][col(kk + 1, nn)] = rb[p].y;
        Bs[buf][kk + 2][col(kk + 2, nn)] = rb[p].z;
        Bs[buf][kk + 3][col(kk + 3, nn)] = rb[p].w;
      } else {
        const int kk = f / TPR, nn = 4 * (f % TPR);
        *reinterpret_cast<float4*>(&Bs[buf][kk][col(kk, nn)]) = rb[p];
      }
    }
  };
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  int buf = 0;
  if (kbeg < kend) {
    load(kbeg);
    store(0);
  }
  __syncthreads();
  for (int k0 = kbeg; k0 < kend; k0 += BK) {
    const bool more = k0 + BK < kend;
    if (more) load(k0 + BK);       // in flight during this slice's products
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[buf][kk][col(kk, 4 * ty)]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[buf][kk][col(kk, 4 * tx)]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    // the other buffer was last read before the previous barrier
    if (more) store(buf ^ 1);
    __syncthreads();
    buf ^= 1;
  }
  const int n = n0 + 4 * tx;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + 4 * ty + i;
    float* c = C + static_cast<long long>(m) * g.ldc + n;
    if (g.ksplit > 1) {
#pragma unroll
      for (int j = 0; j < 4; ++j) atomicAdd(c + j, g.alpha * acc[i][j]);
    } else {
      float4 old = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (g.beta != 0.0f) old = *reinterpret_cast<const float4*>(c);
      const float ov[4] = {old.x, old.y, old.z, old.w};
      float r[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        r[j] = (g.beta == 0.0f ? g.alpha * acc[i][j] : fmaf(g.alpha, acc[i][j], g.beta * ov[j])) +
               (m == n + j ? g.diag : 0.0f);
      *reinterpret_cast<float4*>(c) = make_float4(r[0], r[1], r[2], r[3]);
    }
  }
}

// ---------------------------------------------------------------------------
// The same product on the tensor cores, for the large GEMMs (M and N multiples
// of 64, K of 32): every fp32 operand x is split into three bf16 parts as it
// is staged into shared memory, hi = bf16(x), mid = bf16(x - hi), lo =
// bf16(x - hi - mid) (both differences exact in fp32), and op(A) op(B) is
// taken as the six products of parts whose orders add up to at most 2^-16
// (lo hi, hi lo, mid mid, mid hi, hi mid, hi hi, smallest first) with
// mma.sync.m16n8k16 (bf16 in, fp32 accumulate).  What is dropped (mid lo, lo
// mid, lo lo and the split's residual) is about 2^-24 of each product, the
// rounding of an fp32 product; with hi and lo only (three products) the
// products kept about 2^-16, which let a 40-step calibration of the value
// objective stall on one head where the float64 oracle falls to half.
// 64 x 64 output tile, 32-deep k-slices (the next slice's fp32 loads in
// flight during the current slice's products), 4 warps of 32 x 32; fragments
// come from shared memory by ldmatrix (the transposing form for an operand
// kept [k][row]).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// hi, mid and lo bf16 parts of x, packed with y's: {lo16 = part of x, hi16 =
// part of y}
__device__ __forceinline__ void split_bf16x2(float x, float y, uint32_t& hi, uint32_t& mid,
                                             uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const float2 hf = __bfloat1622float2(h);
  const float rx = x - hf.x, ry = y - hf.y;
  const __nv_bfloat162 m = __floats2bfloat162_rn(rx, ry);
  const float2 mf = __bfloat1622float2(m);
  const __nv_bfloat162 l = __floats2bfloat162_rn(rx - mf.x, ry - mf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  mid = *reinterpret_cast<const uint32_t*>(&m);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <int TA, int TB>
__global__ void __launch_bounds__(128) gemm_tc_kernel(Gemm g) {
  constexpr int BM = 64, BK = 32;
  // An operand whose k is its contiguous index (A stored M x K, B stored N x K)
  // is kept [row][k] with rows of 40 bf16 (80 B); the other (A stored K x M,
  // B stored K x N) is kept as stored, [k][row] with rows of 72 bf16 (144 B),
  // and read with the transposing ldmatrix.  Both strides put the 8 rows of
  // one ldmatrix in different banks, and every staging store is 8 bytes.
  constexpr int RK = BK + 8, RR = BM + 8, PLANE = BM * RK;
  static_assert(BK * RR <= PLANE, "a [k][row] tile fits a plane");
  __shared__ __align__(16) uint16_t sA[3][PLANE];    // [hi, mid, lo]
  __shared__ __align__(16) uint16_t sB[3][PLANE];
  const int bz = blockIdx.z / g.ksplit, kz = blockIdx.z % g.ksplit;
  const int kbeg = kz * g.kchunk, kend = min(g.K, kbeg + g.kchunk);
  const float* A = g.A + bz * g.sA;
  const float* B = g.B + bz * g.sB;
  float* C = g.C + bz * g.sC;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BM;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = (warp >> 1) * 32, wn = (warp & 1) * 32;
  constexpr bool kA = TA == 0, kB = TB == 1;     // k contiguous in global memory
  float4 ra[4], rb[4];
  // f-th float4 of a 64 x 32 slice: k-contiguous: row f / 8, k 4 (f % 8);
  // row-contiguous: k f / 16, row 4 (f % 16)
  auto load = [&](int k0) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int f = tid + 128 * p;
      ra[p] = kA ? *reinterpret_cast<const float4*>(A + static_cast<long long>(m0 + f / 8) * g.lda +
                                                    k0 + 4 * (f % 8))
                 : *reinterpret_cast<const float4*>(A + static_cast<long long>(k0 + f / 16) * g.lda +
                                                    m0 + 4 * (f % 16));
      rb[p] = kB ? *reinterpret_cast<const float4*>(B + static_cast<long long>(n0 + f / 8) * g.ldb +
                                                    k0 + 4 * (f % 8))
                 : *reinterpret_cast<const float4*>(B + static_cast<long long>(k0 + f / 16) * g.ldb +
                                                    n0 + 4 * (f % 16));
    }
  };
  auto put = [&](uint16_t (*P)[PLANE], const float4& v, int f, bool kfast) {
    const int off = kfast ? (f / 8) * RK + 4 * (f % 8) : (f / 16) * RR + 4 * (f % 16);
    uint32_t h0, m0, l0, h1, m1, l1;
    split_bf16x2(v.x, v.y, h0, m0, l0);
    split_bf16x2(v.z, v.w, h1, m1, l1);
    *reinterpret_cast<uint2*>(P[0] + off) = make_uint2(h0, h1);
    *reinterpret_cast<uint2*>(P[1] + off) = make_uint2(m0, m1);
    *reinterpret_cast<uint2*>(P[2] + off) = make_uint2(l0, l1);
  };
  auto store = [&]() {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int f = tid + 128 * p;
      put(sA, ra[p], f, kA);
      put(sB, rb[p], f, kB);
    }
  };
  float acc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.0f;
  if (kbeg < kend) {
    load(kbeg);
    store();
  }
  __syncthreads();
  // Element offsets this lane gives ldmatrix.  A (m16 x k16 tile at row r0,
  // k ks): matrix j = lane / 8 holds rows 8 (j & 1), k 8 (j >> 1); [row][k]:
  // lane addresses row r0 + lane % 16, k ks + 8 (lane / 16); [k][row]
  // (transposed): k ks + lane % 8 + 8 (lane / 16), row r0 + 8 ((lane / 8) % 2).
  // B (two n8 tiles at row r0): matrix j holds rows 8 (j >> 1), k 8 (j & 1);
  // [row][k]: row r0 + lane % 8 + 8 (lane / 16), k ks + 8 ((lane / 8) % 2);
  // [k][row]: k ks + lane % 8 + 8 ((lane / 8) % 2), row r0 + 8 (lane / 16).
  const int l8 = lane & 7, l16 = lane >> 4, lb = (lane >> 3) & 1;
  auto a_off = [&](int r0, int ks) {
    return kA ? (r0 + (lane & 15)) * RK + ks + 8 * l16 : (ks + l8 + 8 * l16) * RR + r0 + 8 * lb;
  };
  auto b_off = [&](int r0, int ks) {
    return kB ? (r0 + l8 + 8 * l16) * RK + ks + 8 * lb : (ks + l8 + 8 * lb) * RR + r0 + 8 * l16;
  };
  for (int k0 = kbeg; k0 < kend; k0 += BK) {
    const bool more = k0 + BK < kend;
    if (more) load(k0 + BK);
#pragma unroll
    for (int ks = 0; ks < BK; ks += 16) {
      uint32_t af[3][2][4], bf[3][4][2];     // [hi, mid, lo] fragments
#pragma unroll
      for (int pl = 0; pl < 3; ++pl) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const uint32_t ad =
              static_cast<uint32_t>(__cvta_generic_to_shared(sA[pl] + a_off(wm + 16 * mt, ks)));
          if (kA) ldsm_x4(ad, af[pl][mt][0], af[pl][mt][1], af[pl][mt][2], af[pl][mt][3]);
          else ldsm_x4_t(ad, af[pl][mt][0], af[pl][mt][1], af[pl][mt][2], af[pl][mt][3]);
        }
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const uint32_t bd =
              static_cast<uint32_t>(__cvta_generic_to_shared(sB[pl] + b_off(wn + 16 * np, ks)));
          if (kB)
            ldsm_x4(bd, bf[pl][2 * np][0], bf[pl][2 * np][1], bf[pl][2 * np + 1][0],
                    bf[pl][2 * np + 1][1]);
          else
            ldsm_x4_t(bd, bf[pl][2 * np][0], bf[pl][2 * np][1], bf[pl][2 * np + 1][0],
                      bf[pl][2 * np + 1][1]);
        }
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          mma_bf16_acc(acc[mt][nt], af[2][mt], bf[0][nt][0], bf[0][nt][1]);   // lo hi
          mma_bf16_acc(acc[mt][nt], af[0][mt], bf[2][nt][0], bf[2][nt][1]);   // hi lo
          mma_bf16_acc(acc[mt][nt], af[1][mt], bf[1][nt][0], bf[1][nt][1]);   // mid mid
          mma_bf16_acc(acc[mt][nt], af[1][mt], bf[0][nt][0], bf[0][nt][1]);   // mid hi
          mma_bf16_acc(acc[mt][nt], af[0][mt], bf[1][nt][0], bf[1][nt][1]);   // hi mid
          mma_bf16_acc(acc[mt][nt], af[0][mt], bf[0][nt][0], bf[0][nt][1]);   // hi hi
        }
    }
    __syncthreads();              // every warp is done with this slice's planes
    if (more) {
      store();
      __syncthreads();
    }
  }
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int m = m0 + wm + 16 * mt + gq + 8 * hh;
        const int n = n0 + wn + 8 * nt + 2 * tq;
        float* c = C + static_cast<long long>(m) * g.ldc + n;
        const float v0 = acc[mt][nt][2 * hh], v1 = acc[mt][nt][2 * hh + 1];
        if (g.ksplit > 1) {
          atomicAdd(c, g.alpha * v0);
          atomicAdd(c + 1, g.alpha * v1);
        } else {
          float2 old = make_float2(0.0f, 0.0f);
          if (g.beta != 0.0f) old = *reinterpret_cast<const float2*>(c);
          const float r0 = (g.beta == 0.0f ? g.alpha * v0 : fmaf(g.alpha, v0, g.beta * old.x)) +
                           (m == n ? g.diag : 0.0f);
          const float r1 = (g.beta == 0.0f ? g.alpha * v1 : fmaf(g.alpha, v1, g.beta * old.y)) +
                           (m == n + 1 ? g.diag : 0.0f);
          *reinterpret_cast<float2*>(c) = make_float2(r0, r1);
        }
      }
}

// ---------------------------------------------------------------------------
// Row kernels (one warp per row of kD = 128 elements; lane l owns 4l .. 4l+3)
// ---------------------------------------------------------------------------

// INT2 quantiser of the library (fp32 arithmetic, fp16 scale and zero, round
// half to even), row by row, keeping what the straight-through backward needs:
// flag 0 = code not at a clamp, 1 = clamped high (value follows c * max),
// 2 = clamped low (follows c * min); argmax / argmin (first index on ties).
__global__ void quantise_rows_kernel(const float* __restrict__ r, float* __restrict__ rt,
                                     uint8_t* __restrict__ flag, int* __restrict__ amax,
                                     int* __restrict__ amin, long long rows, float clip) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float4 x4 = *reinterpret_cast<const float4*>(r + row * kD + 4 * lane);
  const float x[4] = {x4.x, x4.y, x4.z, x4.w};
  float mx = x[0], mn = x[0];
  int imx = 4 * lane, imn = 4 * lane;
#pragma unroll
  for (int j = 1; j < 4; ++j) {
    if (x[j] > mx) { mx = x[j]; imx = 4 * lane + j; }
    if (x[j] < mn) { mn = x[j]; imn = 4 * lane + j; }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float omx = __shfl_xor_sync(0xffffffffu, mx, off);
    const int oimx = __shfl_xor_sync(0xffffffffu, imx, off);
    const float omn = __shfl_xor_sync(0xffffffffu, mn, off);
    const int oimn = __shfl_xor_sync(0xffffffffu, imn, off);
    if (omx > mx || (omx == mx && oimx < imx)) { mx = omx; imx = oimx; }
    if (omn < mn || (omn == mn && oimn < imn)) { mn = omn; imn = oimn; }
  }
  const float mxc = __fmul_rn(clip, mx);
  const float mnc = __fmul_rn(clip, mn);
  const float s = __half2float(__float2half_rn(__fdiv_rn(__fsub_rn(mxc, mnc), 3.0f)));
  const float z = __half2float(__float2half_rn(mnc));
  float o[4];
  uint32_t fl = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float code = 0.0f;
    uint32_t f = 2;
    if (s != 0.0f) {
      const float t = __fdiv_rn(__fsub_rn(x[j], z), s);
      code = fminf(fmaxf(rintf(t), 0.0f), 3.0f);
      f = t > 3.0f ? 1u : (t < 0.0f ? 2u : 0u);
    }
    o[j] = fmaf(code, s, z);      // code * s is exact: one rounding, as the oracle's
    fl |= f << (8 * j);
  }
  *reinterpret_cast<float4*>(rt + row * kD + 4 * lane) = make_float4(o[0], o[1], o[2], o[3]);
  *reinterpret_cast<uint32_t*>(flag + row * kD + 4 * lane) = fl;
  if (lane == 0) {
    amax[row] = imx;
    amin[row] = imn;
  }
}

// d loss / d r from d loss / d r~: identity where the code is not clamped; the
// clamped elements' gradients, times c, go to the row's argmax / argmin.
__global__ void ste_backward_kernel(const float* __restrict__ grt, const uint8_t* __restrict__ flag,
                                    const int* __restrict__ amax, const int* __restrict__ amin,
                                    float* __restrict__ gr, long long rows, float clip) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float4 g4 = *reinterpret_cast<const float4*>(grt + row * kD + 4 * lane);
  const float g[4] = {g4.x, g4.y, g4.z, g4.w};
  const uint32_t fl = *reinterpret_cast<const uint32_t*>(flag + row * kD + 4 * lane);
  float o[4], sh = 0.0f, sl = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t f = (fl >> (8 * j)) & 0xffu;
    o[j] = f == 0 ? g[j] : 0.0f;
    if (f == 1) sh += g[j];
    if (f == 2) sl += g[j];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    sh += __shfl_xor_sync(0xffffffffu, sh, off);
    sl += __shfl_xor_sync(0xffffffffu, sl, off);
  }
  const int im = amax[row], in = amin[row];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (4 * lane + j == im) o[j] = fmaf(clip, sh, o[j]);
    if (4 * lane + j == in) o[j] = fmaf(clip, sl, o[j]);
  }
  *reinterpret_cast<float4*>(gr + row * kD + 4 * lane) = make_float4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------------------
// Causal softmax over a row of T logits (one CTA per row).  Row q * G + h of a
// head belongs to the query at position T - Nq + q.  mode 0: write p (the
// reference attention).  mode 1: write p~, dp = p~ - p and add the row's
// KL(p || p~) to kl[head].
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  v = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) v = is_max ? fmaxf(v, red[i]) : v + red[i];
  return v;
}

__global__ void softmax_rows_kernel(const float* __restrict__ logits, const float* __restrict__ p,
                                    float* __restrict__ out, float* __restrict__ dp,
                                    float* __restrict__ kl, int T, int Nq, int G, int mode) {
  __shared__ float red[32];
  const int row = blockIdx.x, head = blockIdx.y;
  const long long base = (static_cast<long long>(head) * Nq * G + row) * T;
  const int pos = T - Nq + row / G;
  float mx = -INFINITY;
  for (int t = threadIdx.x; t <= pos; t += blockDim.x) mx = fmaxf(mx, logits[base + t]);
  mx = block_reduce(mx, red, true);
  float sum = 0.0f;
  for (int t = threadIdx.x; t <= pos; t += blockDim.x) sum += __expf(logits[base + t] - mx);
  sum = block_reduce(sum, red, false);
  const float inv = 1.0f / sum, lsum = logf(sum);
  float klp = 0.0f;
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    float v = 0.0f;
    if (t <= pos) v = __expf(logits[base + t] - mx) * inv;
    out[base + t] = v;
    if (mode == 1) {
      const float pr = p[base + t];
      dp[base + t] = v - pr;
      if (pr > 0.0f) klp += pr * (logf(pr) - (logits[base + t] - mx - lsum));
    }
  }
  if (mode == 1) {
    klp = block_reduce(klp, red, false);
    if (threadIdx.x == 0) atomicAdd(kl + head, klp);
  }
}

// d loss / d logit = p~ (g - <p~, g>) + (p~ - p) / Nq  (the KL part only with
// with_kl).  In place over g.
__global__ void softmax_backward_kernel(const float* __restrict__ pt, const float* __restrict__ p,
                                        float* __restrict__ g, int T, int Nq, int G, float inv_nq,
                                        int with_kl) {
  __shared__ float red[32];
  const int row = blockIdx.x, head = blockIdx.y;
  const long long base = (static_cast<long long>(head) * Nq * G + row) * T;
  float dot = 0.0f;
  for (int t = threadIdx.x; t < T; t += blockDim.x) dot = fmaf(pt[base + t], g[base + t], dot);
  dot = block_reduce(dot, red, false);
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    const float a = pt[base + t];
    float v = a * (g[base + t] - dot);
    if (with_kl) v = fmaf(a - p[base + t], inv_nq, v);
    g[base + t] = v;
  }
}

// err[head] += sum e^2 over the head's Nq x Dm block; ge = coef * e.
__global__ void sq_err_kernel(const float* __restrict__ e, float* __restrict__ ge,
                              float* __restrict__ err, long long n, float coef) {
  __shared__ float red[32];
  const int head = blockIdx.y;
  const float* eh = e + head * n;
  float* gh = ge + head * n;
  float s = 0.0f;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float v = eh[i];
    s = fmaf(v, v, s);
    gh[i] = coef * v;
  }
  s = block_reduce(s, red, false);
  if (threadIdx.x == 0) atomicAdd(err + head, s);
}

// ---------------------------------------------------------------------------
// Element kernels
// ---------------------------------------------------------------------------

// out = bf16 x (- mu per column when mu != null), fp32.
__global__ void bf16_to_f32_kernel(const uint16_t* __restrict__ x, const float* __restrict__ mu,
                                   float* __restrict__ out, long long rows_per_head, long long n) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float v = __uint_as_float(static_cast<uint32_t>(x[i]) << 16);
    if (mu) v = __fsub_rn(v, mu[(i / (rows_per_head * kD)) * kD + (i % kD)]);
    out[i] = v;
  }
}

// y = x + mu per column (per head)
__global__ void add_mu_kernel(float* __restrict__ x, const float* __restrict__ mu,
                              long long rows_per_head, long long n) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    x[i] += mu[(i / (rows_per_head * kD)) * kD + (i % kD)];
}

// S = A - A^T (kD x kD per head)
__global__ void skew_kernel(const float* __restrict__ A, float* __restrict__ S, int heads) {
  const long long total = static_cast<long long>(heads) * kD * kD;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long h = i / (kD * kD), k = i % (kD * kD);
    const int r = static_cast<int>(k / kD), c = static_cast<int>(k % kD);
    S[i] = A[h * kD * kD + r * kD + c] - A[h * kD * kD + c * kD + r];
  }
}

// out = s * f_h * op(X) + d * I for kD x kD matrices (op = transpose when tr);
// f_h = hf[2 h] if hf != nullptr, else 1; head strides sx, so (in floats)
__global__ void scale_kernel(const float* __restrict__ X, long long sx, int tr, float* __restrict__ out,
                             long long so, float s, float d, int heads,
                             const float* __restrict__ hf = nullptr) {
  const long long total = static_cast<long long>(heads) * kD * kD;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long h = i / (kD * kD), k = i % (kD * kD);
    const int r = static_cast<int>(k / kD), c = static_cast<int>(k % kD);
    const float x = X[h * sx + (tr ? c * kD + r : r * kD + c)];
    const float sh = hf ? s * hf[2 * h] : s;
    out[h * so + r * kD + c] = sh * x + (r == c ? d : 0.0f);
  }
}

// gA = V - V^T (kD x kD per head, V with head stride sv)
__global__ void skew_of_kernel(const float* __restrict__ V, long long sv, float* __restrict__ gA,
                               int heads) {
  const long long total = static_cast<long long>(heads) * kD * kD;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long h = i / (kD * kD), k = i % (kD * kD);
    const int r = static_cast<int>(k / kD), c = static_cast<int>(k % kD);
    gA[i] = V[h * sv + r * kD + c] - V[h * sv + c * kD + r];
  }
}

// 1-norms (max over columns of sum |.|) per head of X and, if Y != nullptr, of
// Y, into norm[2 head] and norm[2 head + 1] as int bits (non-negative floats
// order like their bit patterns).  One CTA of 1024 threads per head: thread
// (q, c) sums 16 rows of column c.
__global__ void __launch_bounds__(1024) norm1_kernel(const float* __restrict__ X,
                                                     const float* __restrict__ Y, long long sxy,
                                                     unsigned int* __restrict__ norm) {
  __shared__ float part[2][8][kD];
  const int h = blockIdx.y, c = threadIdx.x % kD, q = threadIdx.x / kD;
  const float* Xh = X + h * sxy;
  const float* Yh = Y ? Y + h * sxy : nullptr;
  float sx = 0.0f, sy = 0.0f;
#pragma unroll
  for (int r = 16 * q; r < 16 * q + 16; ++r) {
    sx += fabsf(Xh[r * kD + c]);
    if (Yh) sy += fabsf(Yh[r * kD + c]);
  }
  part[0][q][c] = sx;
  part[1][q][c] = sy;
  __syncthreads();
  if (q < 2) {
    float t = 0.0f;
#pragma unroll
    for (int u = 0; u < 8; ++u) t += part[q][u][c];
    atomicMax(norm + 2 * h + q, __float_as_uint(t));
  }
}

// Per head, the power of two c = 2^-k (k >= 0) with c |Y|_1 <= 1/4 from the
// 1-norms of norm1_kernel: dscale[2h] = c, dscale[2h + 1] = 1/c.
__global__ void dir_scale_kernel(const unsigned int* __restrict__ norm, float* __restrict__ dscale,
                                 int heads) {
  const int h = threadIdx.x;
  if (h >= heads) return;
  const float ny = __uint_as_float(norm[2 * h + 1]);
  int k = 0;
  while (ldexpf(ny, -k) > 0.25f && k < 120) ++k;
  dscale[2 * h] = ldexpf(1.0f, -k);
  dscale[2 * h + 1] = ldexpf(1.0f, k);
}

// out = sum_i c[i] in[i] (+ d I on the first kD x kD block of each head), over
// `len` floats per head at head stride `stride` (inputs and output alike)
struct LinComb {
  const float* in[5];
  float c[5];
  int n;
  float d;
  float* out;
  long long stride;
  int len;
};

__global__ void lincomb_kernel(LinComb L, int heads) {
  const long long total = static_cast<long long>(heads) * L.len;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long h = i / L.len;
    const int k = static_cast<int>(i % L.len);
    const long long at = h * L.stride + k;
    float v = (k < kD * kD && k / kD == k % kD) ? L.d : 0.0f;
    for (int t = 0; t < L.n; ++t) v = fmaf(L.c[t], L.in[t][at], v);
    L.out[at] = v;
  }
}

__global__ void adam_kernel(float* __restrict__ A, const float* __restrict__ g,
                            float* __restrict__ m, float* __restrict__ v, long long n, float lr,
                            float bc1, float bc2) {
  const float b1 = 0.9f, b2 = 0.999f, eps = 1e-8f;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float gi = g[i];
    const float mi = b1 * m[i] + (1.0f - b1) * gi;
    const float vi = b2 * v[i] + (1.0f - b2) * gi * gi;
    m[i] = mi;
    v[i] = vi;
    A[i] -= lr * (mi / bc1) / (sqrtf(vi / bc2) + eps);
  }
}

// hist[head] = (kl[head] + lam * err[head]) / Nq; then clear kl, err
__global__ void loss_kernel(float* __restrict__ kl, float* __restrict__ err, float* __restrict__ hist,
                            int heads, float lam, float inv_nq) {
  const int h = threadIdx.x;
  if (h >= heads) return;
  hist[h] = (kl[h] + lam * err[h]) * inv_nq;
  kl[h] = 0.0f;
  err[h] = 0.0f;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
int grid_for(long long n) { return static_cast<int>(std::min<long long>((n + 255) / 256, 4096)); }

struct Ctx {
  cudaStream_t st;
  int H, T, Nq, G, Dm;
  cudaError_t err = cudaSuccess;
  float norm_S = -1.0f;     // max over heads of |S|_1 from the last rotation(), -1 if unknown
  void check() { if (err == cudaSuccess) err = cudaGetLastError(); }
};

// C = alpha op(A) op(B) + beta C + diag I for every head (strides sA, sB, sC
// per head)
void gemm(Ctx& c, const float* A, int ta, long long sA, int lda, const float* B, int tb,
          long long sB, int ldb, float* C, long long sC, int ldc, int M, int N, int K, float alpha,
          float beta, float diag = 0.0f) {
  const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool tiled = M % 32 == 0 && N % 32 == 0 && K % 64 == 0 && lda % 4 == 0 && ldb % 4 == 0 &&
                     ldc % 4 == 0 && sA % 4 == 0 && sB % 4 == 0 && sC % 4 == 0 && a16(A) &&
                     a16(B) && a16(C);
  // Tensor cores (bf16 x 3) for every tiled product with 64-multiple M and N,
  // except the products by a 128 x 128 matrix (N = K = 128): the rotations
  // r = X R, r~ R^T and g_r~ = g_k~ R, whose rounding moves codes across the
  // quantiser's boundaries (the straight-through gradient of a large generator
  // then missed the float64 oracle by 2.7e-3), and the products of the matrix
  // exponentials, whose errors the squarings amplify.  Those stay in fp32.
  const bool tc = tiled && M % 64 == 0 && N % 64 == 0 && K % 32 == 0 && !(N == kD && K == kD);
  // the 64-wide tile where it still gives a full wave of CTAs, else 32
  const int bm = tc ? 64
               : (tiled && M % 64 == 0 && N % 64 == 0 &&
                  static_cast<long long>(M / 64) * (N / 64) * c.H >= 152) ? 64
               : tiled ? 32 : 64;
  // Few output tiles and a long K (the T-long reductions): cut K so that the
  // grid covers the GPU; partial products are added atomically (beta 0 or 1).
  const long long tiles = static_cast<long long>((N + bm - 1) / bm) * ((M + bm - 1) / bm) * c.H;
  int ksplit = 1;
  if (diag == 0.0f && tiles < 512 && K >= 1024 && (beta == 0.0f || beta == 1.0f) &&
      (beta == 1.0f || (ldc == N && sC == static_cast<long long>(M) * N))) {
    ksplit = static_cast<int>(std::min<long long>(K / 256, (1024 + tiles - 1) / tiles));
    if (ksplit < 2) ksplit = 1;
  }
  const int kchunk = ksplit > 1 ? ((K + ksplit - 1) / ksplit + 63) / 64 * 64 : K;
  if (ksplit > 1) ksplit = (K + kchunk - 1) / kchunk;
  if (ksplit > 1 && beta == 0.0f && c.err == cudaSuccess)
    c.err = cudaMemsetAsync(C, 0, static_cast<size_t>(c.H) * M * N * sizeof(float), c.st);
  Gemm g{A, B, C, M, N, K, lda, ldb, ldc, sA, sB, sC, alpha, beta, ta, tb, ksplit, kchunk, diag};
  dim3 grid((N + bm - 1) / bm, (M + bm - 1) / bm, c.H * ksplit);
  if (tc) {
    if (ta == 0 && tb == 0)
      gemm_tc_kernel<0, 0><<<grid, 128, 0, c.st>>>(g);
    else if (ta == 0)
      gemm_tc_kernel<0, 1><<<grid, 128, 0, c.st>>>(g);
    else if (tb == 0)
      gemm_tc_kernel<1, 0><<<grid, 128, 0, c.st>>>(g);
    else
      gemm_tc_kernel<1, 1><<<grid, 128, 0, c.st>>>(g);
  } else if (!tiled)
    gemm_kernel<<<grid, 256, 0, c.st>>>(g);
  else if (bm == 64)
    gemm_tile_kernel<64, 32><<<grid, 256, 0, c.st>>>(g);
  else
    gemm_tile_kernel<32, 64><<<grid, 64, 0, c.st>>>(g);
  c.check();
}

// Workspace carve-up (floats unless noted), all per-head arrays [H][...]
struct Ws {
  float *x32, *r, *rt, *kt, *gkt, *grt, *gr;        // [T][D]
  float *V32;                                       // [T][D]
  float *Q32;                                       // [Nq*G][D]
  float *logit, *pt, *p, *dp;                       // [Nq*G][T]
  float *att, *gatt;                                // [Nq*G][D]
  float *e, *ge;                                    // [Nq][Dm]
  float *A, *m, *v, *S, *E, *R, *gR, *Gb, *gA;      // [D][D]
  float *X2, *P2, *Q2;                              // 4 [D][D] each (expm scratch pairs)
  float *kl, *errsum;                               // [H]
  unsigned int* norm;                               // [2H]
  float* dscale;                                    // [2H] direction scale and its inverse
  uint8_t* flag;                                    // [T][D]
  int *amax, *amin;                                 // [T]
  size_t total;
};

Ws carve(uint8_t* base, int H, int T, int Nq, int G, int Dm) {
  Ws w;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? base + o : nullptr;
    o += (bytes + 255) & ~static_cast<size_t>(255);
    return p;
  };
  const size_t hd = static_cast<size_t>(H);
  const size_t TD = hd * T * kD * 4, QD = hd * Nq * G * kD * 4, QT = hd * Nq * G * T * 4;
  const size_t DD = hd * kD * kD * 4, D2 = hd * 4 * kD * kD * 4;
  w.x32 = reinterpret_cast<float*>(take(TD));
  w.r = reinterpret_cast<float*>(take(TD));
  w.rt = reinterpret_cast<float*>(take(TD));
  w.kt = reinterpret_cast<float*>(take(TD));
  w.gkt = reinterpret_cast<float*>(take(TD));
  w.grt = reinterpret_cast<float*>(take(TD));
  w.gr = reinterpret_cast<float*>(take(TD));
  w.V32 = reinterpret_cast<float*>(take(TD));
  w.Q32 = reinterpret_cast<float*>(take(QD));
  w.logit = reinterpret_cast<float*>(take(QT));
  w.pt = reinterpret_cast<float*>(take(QT));
  w.p = reinterpret_cast<float*>(take(QT));
  w.dp = reinterpret_cast<float*>(take(QT));
  w.att = reinterpret_cast<float*>(take(QD));
  w.gatt = reinterpret_cast<float*>(take(QD));
  w.e = reinterpret_cast<float*>(take(hd * Nq * Dm * 4));
  w.ge = reinterpret_cast<float*>(take(hd * Nq * Dm * 4));
  w.A = reinterpret_cast<float*>(take(DD));
  w.m = reinterpret_cast<float*>(take(DD));
  w.v = reinterpret_cast<float*>(take(DD));
  w.S = reinterpret_cast<float*>(take(DD));
  w.E = reinterpret_cast<float*>(take(DD));
  w.R = reinterpret_cast<float*>(take(DD));
  w.gR = reinterpret_cast<float*>(take(DD));
  w.Gb = reinterpret_cast<float*>(take(DD));
  w.gA = reinterpret_cast<float*>(take(DD));
  w.X2 = reinterpret_cast<float*>(take(D2));
  w.P2 = reinterpret_cast<float*>(take(D2));
  w.Q2 = reinterpret_cast<float*>(take(D2));
  w.kl = reinterpret_cast<float*>(take(hd * 4));
  w.errsum = reinterpret_cast<float*>(take(hd * 4));
  w.norm = reinterpret_cast<unsigned int*>(take(hd * 8));
  w.dscale = reinterpret_cast<float*>(take(hd * 8));
  w.flag = take(hd * T * kD);
  w.amax = reinterpret_cast<int*>(take(hd * T * 4));
  w.amin = reinterpret_cast<int*>(take(hd * T * 4));
  w.total = o;
  return w;
}

// exp(M) for every head (kD x kD): scaling by 2^j with |M / 2^j|_1 <= 1/2, the
// degree-8 Taylor polynomial of exp(X) - I (truncation error <= 0.5^9 / 9! ~
// 5e-9, below fp32 rounding) by Paterson-Stockmeyer, F = B0 + X^4 B1 with
// B0 = X + X^2/2 + X^3/6, B1 = I/24 + X/120 + X^2/720 + X^3/5040 + X^4/40320
// (4 matrix products), then j squarings.  The squarings carry F = exp(X) - I
// (F <- 2F + F F), so rounding errors stay relative to F rather than to I: the
// rotation stays orthogonal to fp32 accuracy.
//
// With Mb != nullptr the same is done for the block matrix [[M, Mb], [0, M]],
// kept as the pair (u, v) of its diagonal and upper-right blocks: products of
// such matrices stay of that form, (u1, v1)(u2, v2) = (u1 u2, u1 v2 + v1 u2), so
// each product is three kD x kD products instead of one of twice the size.
// Then `out` receives the upper-right block of the exponential, the Frechet
// derivative of exp at M in the direction Mb.  That block is linear in Mb, so
// Mb enters scaled by a power of two c_h with c_h |Mb_h|_1 <= 1/4 (chosen on the
// device) and the result is divided by c_h: the direction does not add
// squarings.
//
// M (or its transpose, trM) and Mb have head stride kD * kD; the scratch pairs
// live in the (4 kD^2 per head) buffers X2, P2, Q2.  The number of squarings
// comes from the 1-norm of M, read on the host (a stream synchronisation)
// except for the adjoint's M = S^T right after the forward exponential of the
// same S, whose norm is remembered in c.norm_S.
void expm(Ctx& c, Ws& w, const float* M, int trM, const float* Mb, float* out) {
  if (c.err != cudaSuccess) return;
  const long long DD = static_cast<long long>(kD) * kD, S4 = 4 * DD;
  const bool pair = Mb != nullptr;
  c.err = cudaMemsetAsync(w.norm, 0, 2 * c.H * sizeof(unsigned int), c.st);
  norm1_kernel<<<dim3(1, c.H), 8 * kD, 0, c.st>>>(M, Mb, DD, w.norm);
  // the direction's per-head scale c_h (c_h |Mb_h|_1 <= 1/4) is set on the device
  if (pair) dir_scale_kernel<<<1, 64, 0, c.st>>>(w.norm, w.dscale, c.H);
  c.check();
  float nmax = 0.0f;
  if (pair && c.norm_S >= 0.0f) {
    // M = S^T and |S^T|_1 = |S|_1 (S is skew), known from this step's forward
    // exponential: no host read needed, the block matrix's norm is at most
    // |S|_1 + 1/4
    nmax = c.norm_S + 0.25f;
  } else {
    std::vector<unsigned int> nb(2 * c.H);
    if (c.err == cudaSuccess)
      c.err = cudaMemcpyAsync(nb.data(), w.norm, 2 * c.H * sizeof(unsigned int),
                              cudaMemcpyDeviceToHost, c.st);
    if (c.err == cudaSuccess) c.err = cudaStreamSynchronize(c.st);
    if (c.err != cudaSuccess) return;
    for (int h = 0; h < c.H; ++h) {
      float f;
      memcpy(&f, &nb[2 * h], 4);
      nmax = std::max(nmax, f);
    }
    if (!pair) c.norm_S = trM ? -1.0f : nmax;
    if (pair) nmax += 0.25f;
  }
  int j = 0;
  while (nmax / ldexpf(1.0f, j) > 0.5f && j < 60) ++j;
  const float sc = ldexpf(1.0f, -j);
  const int g = grid_for(c.H * DD), g2 = grid_for(c.H * 2 * DD);
  const int len = pair ? 2 * static_cast<int>(DD) : static_cast<int>(DD);
  // pairs: X, X^2 in X2; X^3, X^4 in P2; B0 (then F), B1 in Q2
  float* X1 = w.X2;
  float* X2p = w.X2 + 2 * DD;
  float* X3 = w.P2;
  float* X4 = w.P2 + 2 * DD;
  float* F = w.Q2;
  float* B1 = w.Q2 + 2 * DD;
  scale_kernel<<<g, 256, 0, c.st>>>(M, DD, trM, X1, S4, sc, 0.0f, c.H);             // X = M / 2^j
  if (pair) scale_kernel<<<g, 256, 0, c.st>>>(Mb, DD, 0, X1 + DD, S4, sc, 0.0f, c.H, w.dscale);
  c.check();
  // C = alpha A B + beta C (+ diag I on u), A B as pairs when `pair`
  auto prod = [&](const float* A, const float* B, float* C, float alpha, float beta, float diag) {
    gemm(c, A, 0, S4, kD, B, 0, S4, kD, C, S4, kD, kD, kD, kD, alpha, beta, diag);
    if (pair) {
      gemm(c, A, 0, S4, kD, B + DD, 0, S4, kD, C + DD, S4, kD, kD, kD, kD, alpha, beta);
      gemm(c, A + DD, 0, S4, kD, B, 0, S4, kD, C + DD, S4, kD, kD, kD, kD, alpha, 1.0f);
    }
  };
  auto lincomb = [&](float* o, std::initializer_list<std::pair<const float*, float>> terms, float d) {
    LinComb L{};
    L.n = 0;
    for (const auto& t : terms) {
      L.in[L.n] = t.first;
      L.c[L.n] = t.second;
      ++L.n;
    }
    L.d = d;
    L.out = o;
    L.stride = S4;
    L.len = len;
    lincomb_kernel<<<pair ? g2 : g, 256, 0, c.st>>>(L, c.H);
    c.check();
  };
  prod(X1, X1, X2p, 1.0f, 0.0f, 0.0f);                                              // X^2
  prod(X2p, X1, X3, 1.0f, 0.0f, 0.0f);                                              // X^3
  prod(X2p, X2p, X4, 1.0f, 0.0f, 0.0f);                                             // X^4
  lincomb(F, {{X1, 1.0f}, {X2p, 1.0f / 2}, {X3, 1.0f / 6}}, 0.0f);
  lincomb(B1, {{X1, 1.0f / 120}, {X2p, 1.0f / 720}, {X3, 1.0f / 5040}, {X4, 1.0f / 40320}},
          1.0f / 24);
  prod(X4, B1, F, 1.0f, 1.0f, 0.0f);                                                // F = B0 + X^4 B1
  float* cur = F;
  float* nxt = B1;
  for (int s = 0; s < j && c.err == cudaSuccess; ++s) {
    // F <- 2F + F F: (u, v) <- (2u + u u, 2v + u v + v u)
    c.err = cudaMemcpy2DAsync(nxt, S4 * sizeof(float), cur, S4 * sizeof(float), len * sizeof(float), c.H,
                              cudaMemcpyDeviceToDevice, c.st);
    prod(cur, cur, nxt, 1.0f, 2.0f, 0.0f);
    std::swap(cur, nxt);
  }
  if (pair)   // undo the direction's scale
    scale_kernel<<<g, 256, 0, c.st>>>(cur + DD, S4, 0, out, DD, 1.0f, 0.0f, c.H, w.dscale + 1);
  else
    scale_kernel<<<g, 256, 0, c.st>>>(cur, S4, 0, out, DD, 1.0f, 1.0f, c.H);        // F + I
  c.check();
}

// R = R0 exp(A - A^T) for every head; also leaves S and E.
void rotation(Ctx& c, Ws& w, const float* R0) {
  const long long DD = static_cast<long long>(kD) * kD;
  skew_kernel<<<grid_for(c.H * DD), 256, 0, c.st>>>(w.A, w.S, c.H);
  c.check();
  expm(c, w, w.S, 0, nullptr, w.E);
  gemm(c, R0, 0, DD, kD, w.E, 0, DD, kD, w.R, DD, kD, kD, kD, kD, 1.0f, 0.0f);
}

// d loss / dA from d loss / dR (in w.gR): Gb = R0^T gR, then the Frechet
// adjoint L_exp(S^T, Gb) (upper-right block of exp([[S^T, Gb], [0, S^T]])),
// whose skew part is the gradient.
void rotation_backward(Ctx& c, Ws& w, const float* R0) {
  const long long DD = static_cast<long long>(kD) * kD;
  gemm(c, R0, 1, DD, kD, w.gR, 0, DD, kD, w.Gb, DD, kD, kD, kD, kD, 1.0f, 0.0f);
  expm(c, w, w.S, 1, w.Gb, w.Gb);      // Gb is read once, at the start
  skew_of_kernel<<<grid_for(c.H * DD), 256, 0, c.st>>>(w.Gb, DD, w.gA, c.H);
  c.check();
}

// Problem description shared by the entry points.
struct Prob {
  int H, T, Nq, G, Dm;
  const uint16_t *K, *V, *Q;
  const float *W, *R0, *mu;
  float clip_k, clip_v, lambda_k, sm_scale;
};

// Inputs to fp32 (centred keys, values, queries) and the reference attention p
// of the exact keys.
void prepare(Ctx& c, Ws& w, const Prob& pb) {
  const long long TD = static_cast<long long>(pb.T) * kD, QG = static_cast<long long>(pb.Nq) * pb.G;
  const long long QT = QG * pb.T, QD = QG * kD;
  bf16_to_f32_kernel<<<grid_for(pb.H * TD), 256, 0, c.st>>>(pb.K, pb.mu, w.x32, pb.T, pb.H * TD);
  bf16_to_f32_kernel<<<grid_for(pb.H * TD), 256, 0, c.st>>>(pb.V, nullptr, w.V32, pb.T, pb.H * TD);
  bf16_to_f32_kernel<<<grid_for(pb.H * QD), 256, 0, c.st>>>(pb.Q, nullptr, w.Q32, QG, pb.H * QD);
  bf16_to_f32_kernel<<<grid_for(pb.H * TD), 256, 0, c.st>>>(pb.K, nullptr, w.kt, pb.T, pb.H * TD);
  c.check();
  if (c.err == cudaSuccess) c.err = cudaMemsetAsync(w.kl, 0, pb.H * 4, c.st);
  if (c.err == cudaSuccess) c.err = cudaMemsetAsync(w.errsum, 0, pb.H * 4, c.st);
  gemm(c, w.Q32, 0, QD, kD, w.kt, 1, TD, kD, w.logit, QT, pb.T, static_cast<int>(QG), pb.T, kD,
       pb.sm_scale, 0.0f);
  softmax_rows_kernel<<<dim3(static_cast<unsigned>(QG), pb.H), 256, 0, c.st>>>(
      w.logit, nullptr, w.p, nullptr, nullptr, pb.T, pb.Nq, pb.G, 0);
  c.check();
}

// One evaluation of objective `which` (0 keys, 1 values) at the generator in
// w.A: the loss per head into loss[H], and with `grad` d loss / dA into w.gA.
// Keys leave their quantised-key attention p~ in w.pt, which the value
// objective reads.
void objective(Ctx& c, Ws& w, const Prob& pb, int which, bool grad, float* loss) {
  const int H = pb.H, T = pb.T, Nq = pb.Nq, Dm = pb.Dm;
  const long long TD = static_cast<long long>(T) * kD, DD = static_cast<long long>(kD) * kD;
  const long long QG = static_cast<long long>(Nq) * pb.G, QT = QG * T, QD = QG * kD;
  const long long ED = static_cast<long long>(Nq) * Dm, GD = static_cast<long long>(pb.G) * kD;
  const float inv_nq = 1.0f / Nq;
  const float* R0w = pb.R0 + (which ? H * DD : 0);
  const float clip = which ? pb.clip_v : pb.clip_k;
  const float* X = which ? w.V32 : w.x32;          // the rows that are rotated
  const long long rows = static_cast<long long>(H) * T;
  const int row_blocks = static_cast<int>((rows + 7) / 8);
  const float lam = which ? 1.0f : pb.lambda_k;
  // ---- forward
  rotation(c, w, R0w);
  gemm(c, X, 0, TD, kD, w.R, 0, DD, kD, w.r, TD, kD, T, kD, kD, 1.0f, 0.0f);     // r = X R
  quantise_rows_kernel<<<row_blocks, 256, 0, c.st>>>(w.r, w.rt, w.flag, w.amax, w.amin, rows, clip);
  c.check();
  gemm(c, w.rt, 0, TD, kD, w.R, 1, DD, kD, w.kt, TD, kD, T, kD, kD, 1.0f, 0.0f);  // rt R^T
  if (which == 0) {
    add_mu_kernel<<<grid_for(H * TD), 256, 0, c.st>>>(w.kt, pb.mu, T, H * TD);
    c.check();
    gemm(c, w.Q32, 0, QD, kD, w.kt, 1, TD, kD, w.logit, QT, T, static_cast<int>(QG), T, kD,
         pb.sm_scale, 0.0f);
    softmax_rows_kernel<<<dim3(static_cast<unsigned>(QG), H), 256, 0, c.st>>>(
        w.logit, w.p, w.pt, w.dp, w.kl, T, Nq, pb.G, 1);
    c.check();
    gemm(c, w.dp, 0, QT, T, w.V32, 0, TD, kD, w.att, QD, kD, static_cast<int>(QG), kD, T, 1.0f,
         0.0f);                                                                    // dp V
  } else {
    // att = p~ (v~ - v)
    gemm(c, w.pt, 0, QT, T, w.kt, 0, TD, kD, w.att, QD, kD, static_cast<int>(QG), kD, T, 1.0f, 0.0f);
    gemm(c, w.pt, 0, QT, T, w.V32, 0, TD, kD, w.att, QD, kD, static_cast<int>(QG), kD, T, -1.0f,
         1.0f);
  }
  // e = att (Nq x G D) W^T (G D x Dm)
  gemm(c, w.att, 0, QD, static_cast<int>(GD), pb.W, 1, static_cast<long long>(Dm) * GD,
       static_cast<int>(GD), w.e, ED, Dm, Nq, Dm, static_cast<int>(GD), 1.0f, 0.0f);
  sq_err_kernel<<<dim3(std::max(1, std::min(64, static_cast<int>((ED + 255) / 256))), H), 256, 0,
                  c.st>>>(w.e, w.ge, w.errsum, ED, 2.0f * lam * inv_nq);
  c.check();
  loss_kernel<<<1, 64, 0, c.st>>>(w.kl, w.errsum, loss, H, lam, inv_nq);
  c.check();
  if (!grad) return;
  // ---- backward
  // gatt = ge W  (Nq x Dm)(Dm x G D)
  gemm(c, w.ge, 0, ED, Dm, pb.W, 0, static_cast<long long>(Dm) * GD, static_cast<int>(GD), w.gatt,
       QD, static_cast<int>(GD), Nq, static_cast<int>(GD), Dm, 1.0f, 0.0f);
  if (which == 0) {
    // g_pt = gatt V^T (QG x T) in logit's buffer, then the softmax backward
    gemm(c, w.gatt, 0, QD, kD, w.V32, 1, TD, kD, w.logit, QT, T, static_cast<int>(QG), T, kD, 1.0f,
         0.0f);
    softmax_backward_kernel<<<dim3(static_cast<unsigned>(QG), H), 256, 0, c.st>>>(
        w.pt, w.p, w.logit, T, Nq, pb.G, inv_nq, 1);
    c.check();
    // g_kt = scale g_logit^T Q  (T x D)
    gemm(c, w.logit, 1, QT, T, w.Q32, 0, QD, kD, w.gkt, TD, kD, T, kD, static_cast<int>(QG),
         pb.sm_scale, 0.0f);
  } else {
    // g_vt = p~^T gatt  (T x D)
    gemm(c, w.pt, 1, QT, T, w.gatt, 0, QD, kD, w.gkt, TD, kD, T, kD, static_cast<int>(QG), 1.0f,
         0.0f);
  }
  gemm(c, w.gkt, 0, TD, kD, w.R, 0, DD, kD, w.grt, TD, kD, T, kD, kD, 1.0f, 0.0f);   // g_rt
  gemm(c, w.gkt, 1, TD, kD, w.rt, 0, TD, kD, w.gR, DD, kD, kD, kD, T, 1.0f, 0.0f);    // gkt^T rt
  ste_backward_kernel<<<row_blocks, 256, 0, c.st>>>(w.grt, w.flag, w.amax, w.amin, w.gr, rows, clip);
  c.check();
  gemm(c, X, 1, TD, kD, w.gr, 0, TD, kD, w.gR, DD, kD, kD, kD, T, 1.0f, 1.0f);        // + X^T gr
  rotation_backward(c, w, R0w);
}

}  // namespace

size_t optr_workspace_bytes(int H, int T, int Nq, int G, int Dm) {
  return carve(nullptr, H, T, Nq, G, Dm).total;
}

int optr_calibrate(int H, int T, int Nq, int G, int Dm, const uint16_t* K, const uint16_t* V,
                   const uint16_t* Qb, const float* W, const float* R0, const float* mu,
                   float clip_k, float clip_v, float lambda_k, float lr, int steps, float sm_scale,
                   float* R_out, float* hist, void* workspace, cudaStream_t st) {
  Ctx c;
  c.st = st;
  c.H = H; c.T = T; c.Nq = Nq; c.G = G; c.Dm = Dm;
  Ws w = carve(static_cast<uint8_t*>(workspace), H, T, Nq, G, Dm);
  const Prob pb{H, T, Nq, G, Dm, K, V, Qb, W, R0, mu, clip_k, clip_v, lambda_k, sm_scale};
  const long long DD = static_cast<long long>(kD) * kD;
  prepare(c, w, pb);
  for (int which = 0; which < 2 && c.err == cudaSuccess; ++which) {
    float* hw = hist + static_cast<long long>(which) * (steps + 1) * H;
    if (c.err == cudaSuccess) c.err = cudaMemsetAsync(w.A, 0, H * DD * 4, st);
    if (c.err == cudaSuccess) c.err = cudaMemsetAsync(w.m, 0, H * DD * 4, st);
    if (c.err == cudaSuccess) c.err = cudaMemsetAsync(w.v, 0, H * DD * 4, st);
    for (int step = 0; step <= steps && c.err == cudaSuccess; ++step) {
      // the loss before each update, and after the last one (no gradient then)
      objective(c, w, pb, which, step < steps, hw + static_cast<long long>(step) * H);
      if (step == steps) break;
      adam_kernel<<<grid_for(H * DD), 256, 0, st>>>(w.A, w.gA, w.m, w.v, H * DD, lr,
                                                    1.0f - powf(0.9f, step + 1.0f),
                                                    1.0f - powf(0.999f, step + 1.0f));
      c.check();
    }
    // the calibrated rotation (the last forward ran at the final generator);
    // after the keys, the attention p~ they give stays in w.pt for the values
    if (c.err == cudaSuccess)
      c.err = cudaMemcpyAsync(R_out + static_cast<long long>(which) * H * DD, w.R, H * DD * 4,
                              cudaMemcpyDeviceToDevice, st);
  }
  if (c.err == cudaSuccess) c.err = cudaStreamSynchronize(st);
  return c.err == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

int optr_loss_grad(int H, int T, int Nq, int G, int Dm, const uint16_t* K, const uint16_t* V,
                   const uint16_t* Qb, const float* W, const float* R0, const float* mu,
                   float clip_k, float clip_v, float lambda_k, float sm_scale, const float* A_key,
                   const float* A_value, int which, float* loss, float* grad, void* workspace,
                   cudaStream_t st) {
  Ctx c;
  c.st = st;
  c.H = H; c.T = T; c.Nq = Nq; c.G = G; c.Dm = Dm;
  Ws w = carve(static_cast<uint8_t*>(workspace), H, T, Nq, G, Dm);
  const Prob pb{H, T, Nq, G, Dm, K, V, Qb, W, R0, mu, clip_k, clip_v, lambda_k, sm_scale};
  const long long DD = static_cast<long long>(kD) * kD;
  prepare(c, w, pb);
  if (c.err == cudaSuccess)
    c.err = cudaMemcpyAsync(w.A, A_key, H * DD * 4, cudaMemcpyDeviceToDevice, st);
  // the key objective at A_key (its gradient only when it is the one asked for)
  objective(c, w, pb, 0, which == 0, loss);
  if (which == 1) {
    if (c.err == cudaSuccess)
      c.err = cudaMemcpyAsync(w.A, A_value, H * DD * 4, cudaMemcpyDeviceToDevice, st);
    objective(c, w, pb, 1, true, loss);
  }
  if (c.err == cudaSuccess)
    c.err = cudaMemcpyAsync(grad, w.gA, H * DD * 4, cudaMemcpyDeviceToDevice, st);
  if (c.err == cudaSuccess) c.err = cudaStreamSynchronize(st);
  return c.err == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

}  // namespace kvq
