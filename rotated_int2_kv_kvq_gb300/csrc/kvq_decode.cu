// kvq_decode.cu — split-K decode attention over the paged INT2 cache (and the
// BF16 comparison cache), the log-sum-exp combine with the inverse value
// rotation, and the dequantisation test export.
//
// Method: "Output-Aware Rotation for INT2 KV-Cache Quantization" (pith.science
// review of arXiv 2608.02691).  Decode reads the rotated, centred, quantised
// keys with the rotated query (rotation is orthogonal, "What carries the
// argument" mechanism 1; centring only shifts every logit by q.mu, mechanism 2),
// and reads values back with dequantisation and the inverse rotation (mechanism
// 3), which deployment may fold into W_V / W_O ("If this is right", third item).
// Split-K with a log-sum-exp merge follows the FlashDecoding scheme named as
// the comparison point on "The KV cache goes on a diet", "Crush it to INT2".
//
// How the INT2 kernel maps onto sm_103a
// -------------------------------------
// One CTA = 4 warps = one (split, KV head, sequence).  Each warp streams every
// 4th page of the split through its own ring of shared-memory stages filled by
// 1-D TMA bulk copies (cp.async.bulk, mbarrier completion).  A page record
// (1152 B) holds the 16 tokens' codes in tensor-core fragment order, so each lane
// takes its whole share with one 16-byte shared load and hands the codes to
// mma.sync.m16n8k16 without any shuffling:
//   scores  S[token][col] = Kcode[token][dim] . B[dim][col]     (M = 16 tokens)
//   values  O^T[dim][col] += Vcode^T[dim][token] . P[token][col] (M = 16 dims)
// with col = 2*head + {hi, lo}: each operand that is not a code is split into an
// fp16 high part and an fp16 residual, which keeps products at fp32 accuracy.
// Codes become fp16 operands with one AND: a 2-bit field at bits [2p, 2p+1] of
// a 16-bit half is the subnormal fp16 number code * 2^(2p-24), exactly; the
// power of two is folded into B (scores) or removed in the epilogue (values).
#include "kvq_internal.cuh"

#include <math.h>

namespace kvq {

DecodeWs decode_ws_layout(int batch, int Hkv, int H, int splits, bool int2) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  DecodeWs w;
  size_t o = 0;
  w.qfrag_off = o;
  if (int2) o += up(static_cast<size_t>(batch) * Hkv * kQFragWords * 4);
  w.qmeta_off = o;
  if (int2) o += up(static_cast<size_t>(batch) * Hkv * 8 * 4);
  w.part_off = o;
  o += up(static_cast<size_t>(batch) * H * splits * kPartStride * 4);
  w.total = o;
  return w;
}

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kStagesInt2 = 4;
constexpr int kStagesBf16 = 3;

// ---------------------------------------------------------------------------
// Query preparation: q_rot = q R_K for the G query heads of one (b, kv), then
// the scores' B fragments.  B[row][col] for k-block w holds q_rot[head][16w+row]
// * 2^(e_head) * 2^(beta_w), split into fp16 hi / lo by col parity, where
// 2^e_head brings max|q_rot| into [16, 32) and 2^beta_w cancels the code scale of
// position w (see the file comment).  Per head also: kappa = sm_scale*log2e *
// 2^(14 - e) and zeta = sm_scale*log2e * sum(q_rot).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) qprep_kernel(DecodeArgs a, const float* __restrict__ RK,
                                                    float log2_scale) {
  __shared__ float qs[kMaxG][kDim];
  __shared__ float qr[kMaxG][kDim];
  __shared__ float red_sum[kMaxG][4], red_max[kMaxG][4];
  __shared__ int e_sh[kMaxG];
  const int b = blockIdx.x, kv = blockIdx.y, i = threadIdx.x;
  const int G = a.G;
  const float* R = RK + static_cast<size_t>(kv) * kDim * kDim;
  for (int h = 0; h < kMaxG; ++h) {
    float v = 0.0f;
    if (h < G) {
      const uint16_t bits = a.q[(static_cast<size_t>(b) * a.H + kv * G + h) * kDim + i];
      v = __uint_as_float(static_cast<uint32_t>(bits) << 16);
    }
    qs[h][i] = v;
  }
  __syncthreads();
  float acc[kMaxG] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int j = 0; j < kDim; ++j) {
    const float r = R[j * kDim + i];
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) acc[h] = fmaf(qs[h][j], r, acc[h]);
  }
  const int warp = i >> 5, lane = i & 31;
#pragma unroll
  for (int h = 0; h < kMaxG; ++h) {
    qr[h][i] = acc[h];
    float s = acc[h], m = fabsf(acc[h]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, off);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    }
    if (lane == 0) {
      red_sum[h][warp] = s;
      red_max[h][warp] = m;
    }
  }
  __syncthreads();
  if (i < kMaxG) {
    const int h = i;
    const float s = red_sum[h][0] + red_sum[h][1] + red_sum[h][2] + red_sum[h][3];
    const float m = fmaxf(fmaxf(red_max[h][0], red_max[h][1]), fmaxf(red_max[h][2], red_max[h][3]));
    int e = 0;
    if (m > 0.0f && m < INFINITY) {
      int E;
      frexpf(m, &E);             // m = f * 2^E, f in [0.5, 1)
      e = 5 - E;                 // m * 2^e in [16, 32)
    }
    e_sh[h] = e;
    float* qm = const_cast<float*>(a.qmeta) + (static_cast<size_t>(b) * a.Hkv + kv) * 8;
    qm[2 * h] = (h < G) ? log2_scale * ldexpf(1.0f, 14 - e) : 0.0f;
    qm[2 * h + 1] = (h < G) ? log2_scale * s : 0.0f;
  }
  __syncthreads();
  // 32 lanes x 16 registers; thread i writes registers 4*(i&3) .. +3 of lane i>>2
  const int L = i >> 2, g = L >> 2, t = L & 3;
  const int head = g >> 1, part = g & 1;
  uint32_t* dst = const_cast<uint32_t*>(a.qfrag) + ((static_cast<size_t>(b) * a.Hkv + kv) * 32 + L) * 16;
  uint32_t out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = 4 * (i & 3) + k;
    const int w = r >> 1, which = r & 1;
    const int row = 16 * w + 2 * t + 8 * which;
    const int beta = (w <= 4) ? (10 - 2 * w) : (20 - 2 * w);
    float v[2] = {0.0f, 0.0f};
    if (head < G) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float x = ldexpf(qr[head][row + u], e_sh[head] + beta);
        const __half hi = __float2half_rn(x);
        v[u] = part ? (x - __half2float(hi)) : __half2float(hi);
      }
    }
    out[k] = pack_half2(v[0], v[1]);
  }
  *reinterpret_cast<uint4*>(dst + 4 * (i & 3)) = make_uint4(out[0], out[1], out[2], out[3]);
}

// Per-warp page-id supply: lane j holds the page id of the warp's page 32*blk + j.
struct PageIds {
  int cur, nxt, blk;
};

__device__ __forceinline__ int load_page_id(const int32_t* ptab, int p0, int warp, int count,
                                            int blk, int lane) {
  const int i = 32 * blk + lane;
  return (i < count) ? ptab[p0 + warp + kDecodeWarps * i] : -1;
}

// ---------------------------------------------------------------------------
// Shared epilogue: reduce l and the z-term over the 8 lanes of a head, hand the
// warp's (m, l, o[128]) per head to shared memory, merge the 4 warps and write
// the CTA's split partial.
// ---------------------------------------------------------------------------
struct CtaCombineSmem {
  float o[kDecodeWarps][kMaxG][kDim];
  float m[kDecodeWarps][kMaxG];
  float l[kDecodeWarps][kMaxG];
};

__device__ __forceinline__ void cta_combine_and_store(CtaCombineSmem& cs, const DecodeArgs& a,
                                                      int b, int kv, int split) {
  __syncthreads();
  const int d = threadIdx.x;
  for (int h = 0; h < a.G; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, cs.m[w][h]);
    float L = 0.0f, o = 0.0f;
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) {
        if (cs.m[w][h] == -INFINITY) continue;
        const float f = fast_exp2(cs.m[w][h] - M);
        L = fmaf(f, cs.l[w][h], L);
        o = fmaf(f, cs.o[w][h][d], o);
      }
    }
    float* p = a.part + ((static_cast<size_t>(b) * a.H + kv * a.G + h) * a.splits + split) * kPartStride;
    p[4 + d] = o;
    if (d == 0) {
      p[0] = M;
      p[1] = L;
    }
  }
}

// ---------------------------------------------------------------------------
// INT2 split-K decode kernel.
// ---------------------------------------------------------------------------
struct Int2Smem {
  uint8_t ring[kDecodeWarps][kStagesInt2][kInt2Rec];
  uint64_t bar[kDecodeWarps][kStagesInt2];
  int ids[kDecodeWarps][kStagesInt2];
  CtaCombineSmem comb;
};

__global__ void __launch_bounds__(kDecodeThreads, 4) decode_int2_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Int2Smem& sm = *reinterpret_cast<Int2Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int split = blockIdx.x, kv = blockIdx.y, b = blockIdx.z;

  int seq_len = a.seq_lens[b];
  if (seq_len < 0 || seq_len > a.max_pages * kPage) {
    if (threadIdx.x == 0 && split == 0 && kv == 0) atomicOr(a.status, KVQ_STATUS_BAD_SEQLEN);
    seq_len = 0;
  }
  const int n_pages = (seq_len + kPage - 1) / kPage;
  const int p0 = split * a.chunk_pages;
  const int p1 = min(p0 + a.chunk_pages, n_pages);
  const int count = (p1 - p0 > warp) ? (p1 - p0 - warp + kDecodeWarps - 1) / kDecodeWarps : 0;
  const int32_t* ptab = a.page_table + static_cast<size_t>(b) * a.max_pages;
  const uint8_t* pool_kv = a.pool + static_cast<size_t>(kv) * kInt2Rec;
  const size_t page_stride = static_cast<size_t>(a.Hkv) * kInt2Rec;

  if (lane == 0) {
    for (int s = 0; s < kStagesInt2; ++s) mbar_init(smem_u32(&sm.bar[warp][s]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  PageIds ids;
  ids.blk = 0;
  ids.cur = load_page_id(ptab, p0, warp, count, 0, lane);
  ids.nxt = load_page_id(ptab, p0, warp, count, 1, lane);

  // issue page j of this warp (all lanes call; lane 0 copies)
  auto issue = [&](int j) {
    if ((j >> 5) != ids.blk) {
      ids.blk = j >> 5;
      ids.cur = ids.nxt;
      ids.nxt = load_page_id(ptab, p0, warp, count, ids.blk + 1, lane);
    }
    const int id = __shfl_sync(0xffffffffu, ids.cur, j & 31);
    if (lane == 0) {
      const int slot = j % kStagesInt2;
      const uint32_t bar = smem_u32(&sm.bar[warp][slot]);
      const bool ok = id >= 0 && id < a.num_pool_pages;
      sm.ids[warp][slot] = ok ? id : -1;
      if (ok) {
        mbar_arrive_expect_tx(bar, kInt2Rec);
        bulk_g2s(smem_u32(sm.ring[warp][slot]), pool_kv + static_cast<size_t>(id) * page_stride,
                 kInt2Rec, bar);
      } else {
        atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
        mbar_arrive(bar);
      }
    }
  };
  for (int j = 0; j < kStagesInt2 && j < count; ++j) issue(j);
  __syncwarp();

  // B fragments of the rotated query and the head's logit constants
  uint32_t qf[16];
  {
    const uint4* src = reinterpret_cast<const uint4*>(
        a.qfrag + ((static_cast<size_t>(b) * a.Hkv + kv) * 32 + lane) * 16);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint4 v = src[r];
      qf[4 * r] = v.x; qf[4 * r + 1] = v.y; qf[4 * r + 2] = v.z; qf[4 * r + 3] = v.w;
    }
  }
  const float kappa = a.qmeta[(static_cast<size_t>(b) * a.Hkv + kv) * 8 + 2 * t];
  const float zeta = a.qmeta[(static_cast<size_t>(b) * a.Hkv + kv) * 8 + 2 * t + 1];

  float acc[8][4];
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[mb][k] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f, z_run = 0.0f;

  int i = 0;
  for (; i < count; ++i) {
    const int slot = i % kStagesInt2;
    const uint32_t parity = (i / kStagesInt2) & 1;
    if (!mbar_wait_bounded(smem_u32(&sm.bar[warp][slot]), parity)) {
      if (lane == 0) atomicOr(a.status, KVQ_STATUS_TIMEOUT);
      break;
    }
    const bool page_ok = sm.ids[warp][slot] >= 0;
    const uint8_t* st = sm.ring[warp][slot];
    const uint4 kw = *reinterpret_cast<const uint4*>(st + 16 * lane);
    const uint4 vw = *reinterpret_cast<const uint4*>(st + 512 + 16 * lane);
    const uint4 mt = *reinterpret_cast<const uint4*>(st + 1024 + 16 * g);
    __syncwarp();
    if (i + kStagesInt2 < count) {
      if (lane == 0) fence_proxy_async();
      issue(i + kStagesInt2);
    }
    const int pos0 = (p0 + warp + kDecodeWarps * i) * kPage;
    const bool v0 = page_ok && (pos0 + g < seq_len);
    const bool v1 = page_ok && (pos0 + g + 8 < seq_len);

    // ---- scores: S[16 tokens][8 cols], k-block w = code position w
    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int p = 0; p < 5; ++p) {
      const uint32_t m = 0x00030003u << (2 * p);
      mma_f16(s, kw.x & m, kw.z & m, kw.y & m, kw.w & m, qf[2 * p], qf[2 * p + 1]);
    }
    {
      const uint32_t k0 = kw.x >> 10, k1 = kw.y >> 10, k2 = kw.z >> 10, k3 = kw.w >> 10;
#pragma unroll
      for (int p = 5; p < 8; ++p) {
        const uint32_t m = 0x00030003u << (2 * (p - 5));
        mma_f16(s, k0 & m, k2 & m, k1 & m, k3 & m, qf[2 * p], qf[2 * p + 1]);
      }
    }
    // logit (log2 units) = kappa * s_k * (q.c) + zeta * z_k, tokens g and g+8, head t
    const float l0 = v0 ? fmaf(kappa * half_lo(mt.x), s[0] + s[1], zeta * half_hi(mt.x)) : -INFINITY;
    const float l1 = v1 ? fmaf(kappa * half_lo(mt.y), s[2] + s[3], zeta * half_hi(mt.y)) : -INFINITY;

    // ---- online softmax over the 16 tokens of this page (lanes 4g+t share head t)
    float pm = fmaxf(l0, l1);
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
    if (pm > m_run) {
      const float f = fast_exp2(m_run - pm);
#pragma unroll
      for (int mb = 0; mb < 8; ++mb)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[mb][k] *= f;
      l_run *= f;
      z_run *= f;
      m_run = pm;
    }
    const float p0v = v0 ? fast_exp2(l0 - m_run) : 0.0f;
    const float p1v = v1 ? fast_exp2(l1 - m_run) : 0.0f;
    l_run += p0v + p1v;
    float P0 = 0.0f, P1 = 0.0f;
    if (v0) {
      P0 = p0v * half_lo(mt.z);
      z_run = fmaf(p0v, half_hi(mt.z), z_run);
    }
    if (v1) {
      P1 = p1v * half_lo(mt.w);
      z_run = fmaf(p1v, half_hi(mt.w), z_run);
    }
    // ---- P (scaled by s_v) as B fragments of the value product, hi/lo fp16
    const uint32_t X = pack_half2(P0, P1);
    const uint32_t Y = pack_half2(P0 - half_lo(X), P1 - half_hi(X));
    const int src0 = 4 * (2 * t) + (g >> 1);
    const uint32_t xa = __shfl_sync(0xffffffffu, X, src0);
    const uint32_t ya = __shfl_sync(0xffffffffu, Y, src0);
    const uint32_t xb = __shfl_sync(0xffffffffu, X, src0 + 4);
    const uint32_t yb = __shfl_sync(0xffffffffu, Y, src0 + 4);
    const uint32_t va = (g & 1) ? ya : xa;
    const uint32_t vb = (g & 1) ? yb : xb;
    const uint32_t pb0 = __byte_perm(va, vb, 0x5410);
    const uint32_t pb1 = __byte_perm(va, vb, 0x7632);

    // ---- values: O^T[dims of m-block mb][8 cols] += Vcode^T . P
#pragma unroll
    for (int mb = 0; mb < 5; ++mb) {
      const uint32_t m = 0x00030003u << (2 * mb);
      mma_f16(acc[mb], vw.x & m, vw.y & m, vw.z & m, vw.w & m, pb0, pb1);
    }
    {
      const uint32_t u0 = vw.x >> 10, u1 = vw.y >> 10, u2 = vw.z >> 10, u3 = vw.w >> 10;
#pragma unroll
      for (int mb = 5; mb < 8; ++mb) {
        const uint32_t m = 0x00030003u << (2 * (mb - 5));
        mma_f16(acc[mb], u0 & m, u1 & m, u2 & m, u3 & m, pb0, pb1);
      }
    }
  }
  if (i < count) {
    // A wait gave up: let the copies already issued for this warp land (bounded)
    // before the CTA can exit, so no bulk copy targets freed shared memory.
    for (int j = i + 1; j < count && j < i + kStagesInt2; ++j)
      mbar_wait_bounded(smem_u32(&sm.bar[warp][j % kStagesInt2]), (j / kStagesInt2) & 1);
  }

  // ---- warp epilogue
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
    z_run += __shfl_xor_sync(0xffffffffu, z_run, off);
  }
  if (t < a.G) {
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      const float inv_alpha = (mb <= 4) ? __int_as_float((127 + 24 - 2 * mb) << 23)
                                        : __int_as_float((127 + 34 - 2 * mb) << 23);
      sm.comb.o[warp][t][16 * mb + g] = fmaf(acc[mb][0] + acc[mb][1], inv_alpha, z_run);
      sm.comb.o[warp][t][16 * mb + g + 8] = fmaf(acc[mb][2] + acc[mb][3], inv_alpha, z_run);
    }
    if (g == 0) {
      sm.comb.m[warp][t] = m_run;
      sm.comb.l[warp][t] = l_run;
    }
  }
  cta_combine_and_store(sm.comb, a, b, kv, split);
}

// ---------------------------------------------------------------------------
// BF16 split-K decode kernel (comparison point): same skeleton, bf16 operands
// read straight from the staged page, plain logits q.k * sm_scale.
// ---------------------------------------------------------------------------
struct Bf16Smem {
  uint8_t ring[kDecodeWarps][kStagesBf16][kBf16Rec];
  uint64_t bar[kDecodeWarps][kStagesBf16];
  int ids[kDecodeWarps][kStagesBf16];
  CtaCombineSmem comb;
};

__global__ void __launch_bounds__(kDecodeThreads, 2) decode_bf16_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Bf16Smem& sm = *reinterpret_cast<Bf16Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int split = blockIdx.x, kv = blockIdx.y, b = blockIdx.z;

  int seq_len = a.seq_lens[b];
  if (seq_len < 0 || seq_len > a.max_pages * kPage) {
    if (threadIdx.x == 0 && split == 0 && kv == 0) atomicOr(a.status, KVQ_STATUS_BAD_SEQLEN);
    seq_len = 0;
  }
  const int n_pages = (seq_len + kPage - 1) / kPage;
  const int p0 = split * a.chunk_pages;
  const int p1 = min(p0 + a.chunk_pages, n_pages);
  const int count = (p1 - p0 > warp) ? (p1 - p0 - warp + kDecodeWarps - 1) / kDecodeWarps : 0;
  const int32_t* ptab = a.page_table + static_cast<size_t>(b) * a.max_pages;
  const uint8_t* pool_kv = a.pool + static_cast<size_t>(kv) * kBf16Rec;
  const size_t page_stride = static_cast<size_t>(a.Hkv) * kBf16Rec;

  if (lane == 0) {
    for (int s = 0; s < kStagesBf16; ++s) mbar_init(smem_u32(&sm.bar[warp][s]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  PageIds ids;
  ids.blk = 0;
  ids.cur = load_page_id(ptab, p0, warp, count, 0, lane);
  ids.nxt = load_page_id(ptab, p0, warp, count, 1, lane);
  auto issue = [&](int j) {
    if ((j >> 5) != ids.blk) {
      ids.blk = j >> 5;
      ids.cur = ids.nxt;
      ids.nxt = load_page_id(ptab, p0, warp, count, ids.blk + 1, lane);
    }
    const int id = __shfl_sync(0xffffffffu, ids.cur, j & 31);
    if (lane == 0) {
      const int slot = j % kStagesBf16;
      const uint32_t bar = smem_u32(&sm.bar[warp][slot]);
      const bool ok = id >= 0 && id < a.num_pool_pages;
      sm.ids[warp][slot] = ok ? id : -1;
      if (ok) {
        mbar_arrive_expect_tx(bar, kBf16Rec);
        bulk_g2s(smem_u32(sm.ring[warp][slot]), pool_kv + static_cast<size_t>(id) * page_stride,
                 kBf16Rec, bar);
      } else {
        atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
        mbar_arrive(bar);
      }
    }
  };
  for (int j = 0; j < kStagesBf16 && j < count; ++j) issue(j);
  __syncwarp();

  // B fragments: col g = 2*head + part; part 0 carries q (bf16, exact), part 1 is 0
  uint32_t qf[16];
  {
    const int head = g >> 1;
    const bool use = ((g & 1) == 0) && head < a.G;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        a.q + (static_cast<size_t>(b) * a.H + kv * a.G + (head < a.G ? head : 0)) * kDim);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      qf[2 * w] = use ? qrow[(16 * w + 2 * t) >> 1] : 0u;
      qf[2 * w + 1] = use ? qrow[(16 * w + 2 * t + 8) >> 1] : 0u;
    }
  }
  const float kappa = a.log2_scale;

  float acc[8][4];
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[mb][k] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;

  int i = 0;
  for (; i < count; ++i) {
    const int slot = i % kStagesBf16;
    const uint32_t parity = (i / kStagesBf16) & 1;
    if (!mbar_wait_bounded(smem_u32(&sm.bar[warp][slot]), parity)) {
      if (lane == 0) atomicOr(a.status, KVQ_STATUS_TIMEOUT);
      break;
    }
    const bool page_ok = sm.ids[warp][slot] >= 0;
    const uint8_t* st = sm.ring[warp][slot];
    const int pos0 = (p0 + warp + kDecodeWarps * i) * kPage;
    const bool v0 = page_ok && (pos0 + g < seq_len);
    const bool v1 = page_ok && (pos0 + g + 8 < seq_len);

    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const uint4 kf = *reinterpret_cast<const uint4*>(st + 512 * w + 16 * lane);
      mma_bf16(s, kf.x, kf.y, kf.z, kf.w, qf[2 * w], qf[2 * w + 1]);
    }
    uint4 vf[8];
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
      vf[mb] = *reinterpret_cast<const uint4*>(st + 4096 + 512 * mb + 16 * lane);
    __syncwarp();
    if (i + kStagesBf16 < count) {
      if (lane == 0) fence_proxy_async();
      issue(i + kStagesBf16);
    }
    const float l0 = v0 ? kappa * (s[0] + s[1]) : -INFINITY;
    const float l1 = v1 ? kappa * (s[2] + s[3]) : -INFINITY;
    float pm = fmaxf(l0, l1);
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
    if (pm > m_run) {
      const float f = fast_exp2(m_run - pm);
#pragma unroll
      for (int mb = 0; mb < 8; ++mb)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[mb][k] *= f;
      l_run *= f;
      m_run = pm;
    }
    const float P0 = v0 ? fast_exp2(l0 - m_run) : 0.0f;
    const float P1 = v1 ? fast_exp2(l1 - m_run) : 0.0f;
    l_run += P0 + P1;
    const uint32_t X = pack_bf162(P0, P1);
    const float x0 = __uint_as_float(X << 16), x1 = __uint_as_float(X & 0xffff0000u);
    const uint32_t Y = pack_bf162(P0 - x0, P1 - x1);
    const int src0 = 4 * (2 * t) + (g >> 1);
    const uint32_t xa = __shfl_sync(0xffffffffu, X, src0);
    const uint32_t ya = __shfl_sync(0xffffffffu, Y, src0);
    const uint32_t xb = __shfl_sync(0xffffffffu, X, src0 + 4);
    const uint32_t yb = __shfl_sync(0xffffffffu, Y, src0 + 4);
    const uint32_t va = (g & 1) ? ya : xa;
    const uint32_t vb = (g & 1) ? yb : xb;
    const uint32_t pb0 = __byte_perm(va, vb, 0x5410);
    const uint32_t pb1 = __byte_perm(va, vb, 0x7632);
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
      mma_bf16(acc[mb], vf[mb].x, vf[mb].y, vf[mb].z, vf[mb].w, pb0, pb1);
  }
  if (i < count) {
    for (int j = i + 1; j < count && j < i + kStagesBf16; ++j)
      mbar_wait_bounded(smem_u32(&sm.bar[warp][j % kStagesBf16]), (j / kStagesBf16) & 1);
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
  if (t < a.G) {
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      sm.comb.o[warp][t][16 * mb + g] = acc[mb][0] + acc[mb][1];
      sm.comb.o[warp][t][16 * mb + g + 8] = acc[mb][2] + acc[mb][3];
    }
    if (g == 0) {
      sm.comb.m[warp][t] = m_run;
      sm.comb.l[warp][t] = l_run;
    }
  }
  cta_combine_and_store(sm.comb, a, b, kv, split);
}

// ---------------------------------------------------------------------------
// Log-sum-exp combine of the split partials, then out = o_rot R_V^T.
// One CTA per (b, query head); thread d owns element d.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) combine_kernel(DecodeArgs a, const float* __restrict__ RVt,
                                                      int rotate_out, float* __restrict__ out) {
  __shared__ float os[kDim];
  const int bh = blockIdx.x;
  const int h = bh % a.H, kv = h / a.G;
  const int d = threadIdx.x;
  const float* parts = a.part + static_cast<size_t>(bh) * a.splits * kPartStride;
  float M = -INFINITY;
  for (int j = 0; j < a.splits; ++j) M = fmaxf(M, parts[j * kPartStride]);
  float L = 0.0f, o = 0.0f;
  if (M > -INFINITY) {
    for (int j = 0; j < a.splits; ++j) {
      const float mj = parts[j * kPartStride];
      if (mj == -INFINITY) continue;
      const float f = fast_exp2(mj - M);
      L = fmaf(f, parts[j * kPartStride + 1], L);
      o = fmaf(f, parts[j * kPartStride + 4 + d], o);
    }
  }
  o = (L > 0.0f) ? o / L : 0.0f;
  if (rotate_out) {
    os[d] = o;
    __syncthreads();
    const float* Rt = RVt + static_cast<size_t>(kv) * kDim * kDim;
    float r = 0.0f;
    for (int j = 0; j < kDim; ++j) r = fmaf(os[j], Rt[j * kDim + d], r);
    o = r;
  }
  out[static_cast<size_t>(bh) * kDim + d] = o;
}

// Dequantise positions [start, start+len) of one sequence: CTA per (position,
// KV head), thread d per element, following the record layout of include/kvq.h.
__global__ void __launch_bounds__(128) dequant_kernel(const uint8_t* __restrict__ pool,
                                                      int num_pool_pages,
                                                      const int32_t* __restrict__ page_table,
                                                      int max_pages, int Hkv, int seq, int start,
                                                      float* K_out, float* V_out,
                                                      uint32_t* status) {
  const int i = blockIdx.x, kv = blockIdx.y, d = threadIdx.x;
  const int p = start + i;
  if (p < 0 || p >= max_pages * kPage) {
    if (d == 0) atomicOr(status, KVQ_STATUS_BAD_POS);
    return;
  }
  const int id = page_table[static_cast<size_t>(seq) * max_pages + p / kPage];
  if (id < 0 || id >= num_pool_pages) {
    if (d == 0) atomicOr(status, KVQ_STATUS_BAD_PAGE);
    return;
  }
  const uint8_t* rec = pool + (static_cast<size_t>(id) * Hkv + kv) * kInt2Rec;
  const uint32_t* words = reinterpret_cast<const uint32_t*>(rec);
  const int tau = p % kPage;
  const size_t o = (static_cast<size_t>(i) * Hkv + kv) * kDim + d;
  if (K_out) {
    const int w = d >> 4, r = d & 15, h = r >> 3, t = (r >> 1) & 3, e = r & 1;
    const int L = 4 * (tau & 7) + t, word = 2 * (tau >> 3) + h, bit = 16 * e + 2 * w;
    const uint32_t code = (words[4 * L + word] >> bit) & 3u;
    const uint32_t sz = *reinterpret_cast<const uint32_t*>(rec + 1024 + 16 * (tau & 7) + 4 * (tau >> 3));
    K_out[o] = fmaf(static_cast<float>(code), half_lo(sz), half_hi(sz));
  }
  if (V_out) {
    const int m = d >> 4, r = d & 15, g = r & 7, dh = r >> 3;
    const int t = (tau & 7) >> 1, e = tau & 1, th = tau >> 3;
    const int L = 4 * g + t, word = 2 * th + dh, bit = 16 * e + 2 * m;
    const uint32_t code = (words[128 + 4 * L + word] >> bit) & 3u;
    const uint32_t sz =
        *reinterpret_cast<const uint32_t*>(rec + 1024 + 16 * (tau & 7) + 8 + 4 * (tau >> 3));
    V_out[o] = fmaf(static_cast<float>(code), half_lo(sz), half_hi(sz));
  }
}

// out[c][j][i] = in[c][i][j] for count 128x128 matrices.
__global__ void transpose_kernel(const float* __restrict__ in, float* __restrict__ out) {
  __shared__ float tile[32][33];
  const float* src = in + static_cast<size_t>(blockIdx.z) * kDim * kDim;
  float* dst = out + static_cast<size_t>(blockIdx.z) * kDim * kDim;
  const int bx = blockIdx.x * 32, by = blockIdx.y * 32;
  for (int k = threadIdx.y; k < 32; k += blockDim.y)
    tile[k][threadIdx.x] = src[(by + k) * kDim + bx + threadIdx.x];
  __syncthreads();
  for (int k = threadIdx.y; k < 32; k += blockDim.y)
    dst[(bx + k) * kDim + by + threadIdx.x] = tile[threadIdx.x][k];
}

template <typename Smem, typename Kern>
cudaError_t set_smem_attr(Kern kern) {
  static bool done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(Smem)));
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

}  // namespace

cudaError_t launch_qprep(const DecodeArgs& a, const float* RK, float sm_scale, cudaStream_t st) {
  dim3 grid(a.batch, a.Hkv);
  qprep_kernel<<<grid, 128, 0, st>>>(a, RK, sm_scale * kLog2e);
  return cudaGetLastError();
}

cudaError_t launch_decode_int2(const DecodeArgs& a, cudaStream_t st) {
  cudaError_t e = set_smem_attr<Int2Smem>(decode_int2_kernel);
  if (e != cudaSuccess) return e;
  dim3 grid(a.splits, a.Hkv, a.batch);
  decode_int2_kernel<<<grid, kDecodeThreads, sizeof(Int2Smem), st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t st) {
  cudaError_t e = set_smem_attr<Bf16Smem>(decode_bf16_kernel);
  if (e != cudaSuccess) return e;
  dim3 grid(a.splits, a.Hkv, a.batch);
  decode_bf16_kernel<<<grid, kDecodeThreads, sizeof(Bf16Smem), st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_combine(const DecodeArgs& a, const float* RVt, bool rotate_out, float* out,
                           cudaStream_t st) {
  combine_kernel<<<a.batch * a.H, 128, 0, st>>>(a, RVt, rotate_out ? 1 : 0, out);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const uint8_t* pool, int num_pool_pages, const int32_t* page_table,
                           int max_pages, int Hkv, int seq, int start, int len, float* K_out,
                           float* V_out, uint32_t* status, cudaStream_t st) {
  dim3 grid(len, Hkv);
  dequant_kernel<<<grid, 128, 0, st>>>(pool, num_pool_pages, page_table, max_pages, Hkv, seq,
                                       start, K_out, V_out, status);
  return cudaGetLastError();
}

cudaError_t launch_transpose(const float* in, float* out, int count, cudaStream_t st) {
  dim3 grid(kDim / 32, kDim / 32, count), block(32, 8);
  transpose_kernel<<<grid, block, 0, st>>>(in, out);
  return cudaGetLastError();
}

int decode_int2_ctas_per_sm() {
  if (set_smem_attr<Int2Smem>(decode_int2_kernel) != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_int2_kernel, kDecodeThreads,
                                                    sizeof(Int2Smem)) != cudaSuccess || n < 1)
    return 1;
  return n;
}

int decode_bf16_ctas_per_sm() {
  if (set_smem_attr<Bf16Smem>(decode_bf16_kernel) != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_bf16_kernel, kDecodeThreads,
                                                    sizeof(Bf16Smem)) != cudaSuccess || n < 1)
    return 1;
  return n;
}

}  // namespace kvq
