// Two-call forked Gated DeltaNet on the 5th-generation tensor cores (tcgen05, TF32).
//
// Same chunk form as the warp-MMA kernel (fork_gdn.cu; gated delta rule of the
// rainbus summary "前置知识", chunked solve of the DFlash-TfM summary "GDN을 위한
// 롤백 없는 트리 검증"): with the chunk's start state S0, G_t = sum_{s<=t} log a_s,
// Gamma_ts = exp(G_t - G_s),
//   (I + A) U = diag(eta) (V - diag(e^G) K S0^T),  A_ts = eta_t Gamma_ts k_t.k_s  (s < t)
//   O = diag(e^G) Q S0^T + (tril(Gamma) * Q K^T) U
//   S = e^{G_last} S0 + U^T diag(Gamma_last) K.
// One CTA per (segment, head), d = 128.  The state S (128 x 128 fp32, lane = v
// row) lives in tensor memory for the whole segment and is the accumulator of
// the state update and the A operand of the next chunk's products.  Per chunk
// one thread issues, as kind::tf32 MMAs with f32 accumulation in TMEM:
//   M1  [Q; K] K^T      (A, B: normalised q/k rows in 128-byte-swizzled smem)
//   M3  S [Q; K]^T      (A = S from TMEM)            -> e^G Q S^T, K S^T
//   M4  U^T = R^T T^T   (A = R^T from TMEM, B = T = (I + A)^{-1} in smem)
//   M5  O^T += U^T P^T  (A = U^T from TMEM, B = P in smem)
//   M6  S += U^T diag(Gamma_last) K   (A = U^T from TMEM, B = a Gamma-scaled K^T copy)
// Every operand written by threads is rounded to TF32 (round to nearest) first;
// T is formed in fp32 by blocked forward substitution.  Eight warps: all of
// them stage inputs and run the SIMT steps; each TMEM lane quarter is served by
// two warps (one per column half).  Waits are bounded and agreed CTA-wide.
#include "fork_gdn.cuh"
#include "tc_ptx.cuh"

namespace fork {

namespace {
constexpr int D = 128;
constexpr int C = 64;
constexpr int NT = 256;
constexpr int KW = 4;
constexpr int HR = C + KW - 1;
constexpr int LDC = C + 4;   // plain 64-wide fp32 tiles
constexpr int LDV = D + 4;   // plain 128-wide fp32 tile
constexpr uint32_t kTmemCols = 512;
// TMEM columns
constexpr uint32_t TS = 0, TD1 = 128, TD3 = 192, TR = 320, TU = 384;

struct Lay {
  static constexpr int XQK = 0;                     // [Q;K] 128 rows x 128 fp32, 4 boxes of 32 columns
  static constexpr int TB = XQK + 4 * 16384;        // T as B operand: 64 rows x 64 fp32, 2 boxes
  static constexpr int PB = TB + 2 * 8192;          // P as B operand
  static constexpr int AM = PB + 2 * 8192;          // plain A [64][LDC]
  static constexpr int TM = AM + C * LDC * 4;       // plain T [64][LDC]
  static constexpr int XS = TM + C * LDC * 4;       // inverse scratch [3*256]
  static constexpr int VH = XS + 3 * 256 * 4;       // plain v [64][LDV]; later bf16 output staging
  static constexpr int RAW = VH + C * LDV * 4;      // staged raw rows [3][HR][D] bf16
  static constexpr int GT = RAW + 3 * HR * D * 2;   // gates: ga, ge, G, EG, GL, ETA
  static constexpr int BAR = GT + 6 * C * 4;
  static constexpr int BYTES = BAR + 128;
  static constexpr int SMEM = BYTES + 1024;
};
static_assert(Lay::SMEM <= 232448, "shared memory budget");
static_assert(Lay::AM % 1024 == 0 && Lay::VH - Lay::AM >= 2 * 16384, "K^T copy fits over the inverse's buffers");

enum { B_M1 = 0, B_M3, B_M4, B_M56, B_FIN, B_N };

// SFU approximations (relative error ~2^-22): 2^x, 1/x, 1/sqrt(x)
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcpf(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rsqrtf_(float x) {
  float y;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;
// SiLU(y) = y / (1 + e^-y)
__device__ __forceinline__ float silu(float y) { return y * rcpf(1.f + ex2f(-y * kLog2e)); }

__device__ __forceinline__ uint32_t tf32_bits(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
// byte offset of fp32 element (r, c) in a K-major 128-byte-swizzled tile of
// 32-column boxes of `rows` rows
__device__ __forceinline__ int swz(int rows, int r, int c) {
  const int cc = c & 31;
  return (c >> 5) * rows * 128 + r * 128 + ((((cc >> 2) ^ (r & 7))) << 4) + ((cc & 3) << 2);
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 4 : 0));
}
}  // namespace

template <bool BRANCH>
__global__ void __launch_bounds__(NT, 1) gdn_tc_kernel(const GdnParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int32_t* meta = p.meta;
  const MetaLayout& L = p.L;
  if (meta[H_VALID] == 0) return;
  const int R = meta[H_R];
  const int idx = blockIdx.x;
  int seg, j;
  if (BRANCH) {
    if (idx >= meta[H_NQ]) return;
    seg = R + idx;
    j = meta[L.seg_req + seg];
  } else {
    if (idx >= R) return;
    seg = idx;
    j = idx;
  }
  const int h = blockIdx.y;
  const int H = p.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int start = meta[L.seg_start + seg];
  const int len = meta[L.seg_len + seg];
  const int pos0 = meta[L.seg_pos0 + seg];
  const int pl = meta[L.req_prefix_len + j];
  const int ck = BRANCH ? -1 : meta[L.req_ckpt_pos + j];
  const bool resumed = !BRANCH && pl > 0;
  if (resumed && (!p.state_in || !p.hist_in)) {
    if (tid == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_BAD_PREFIX);
    return;
  }
  const uint16_t* hist = (BRANCH || resumed) ? p.hist_in : nullptr;
  const float* S0 = (BRANCH || resumed) ? p.state_in : nullptr;
  const int64_t state_base = (static_cast<int64_t>(j) * H + h) * D * D;

  unsigned char* xqk = sm + Lay::XQK;
  unsigned char* tb = sm + Lay::TB;
  unsigned char* pb = sm + Lay::PB;
  float* am = reinterpret_cast<float*>(sm + Lay::AM);
  float* tm = reinterpret_cast<float*>(sm + Lay::TM);
  float* xs = reinterpret_cast<float*>(sm + Lay::XS);
  float* vh = reinterpret_cast<float*>(sm + Lay::VH);
  uint16_t* raw_st = reinterpret_cast<uint16_t*>(sm + Lay::RAW);
  float* ga = reinterpret_cast<float*>(sm + Lay::GT);
  float* ge = ga + C;
  float* G = ge + C;
  float* EG = G + C;
  float* GL = EG + C;
  float* ETA = GL + C;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::BAR + B_N * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + Lay::BAR + B_N * 8 + 8);

  if (tid == 0) {
    for (int b = 0; b < B_N; ++b) tc::mbar_init(&bars[b], 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM lane / column-half of this thread
  const int row = (warp & 3) * 32 + lane;
  const int half = warp >> 2;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;

  auto xsrc_of = [&](int st) -> const uint16_t* { return st == 0 ? p.q : (st == 1 ? p.k : p.v); };
  auto raw = [&](int o_seg, int s, int c) -> float {
    if (o_seg >= 0) return bf2f(xsrc_of(s)[(static_cast<int64_t>(start + o_seg) * H + h) * D + c]);
    const int r = KW - 1 + o_seg;
    if (r < 0 || hist == nullptr) return 0.f;
    return bf2f(hist[((static_cast<int64_t>(j * (KW - 1) + r) * 3 + s) * H + h) * D + c]);
  };
  // stage raw rows c0n-3 .. c0n+C-1 (zero beyond the segment) and the gates of a chunk:
  // thread = (16-byte piece, first row); rows step by NT/16
  auto prefetch = [&](int c0n) {
    const int ch = tid & 15, r0 = tid >> 4;
#pragma unroll
    for (int st = 0; st < 3; ++st) {
      for (int r = r0; r < HR; r += NT / 16) {
        const int o_seg = c0n - (KW - 1) + r;
        const uint16_t* src = p.q;
        bool valid = false;
        if (o_seg >= 0 && o_seg < len) {
          src = xsrc_of(st) + (static_cast<int64_t>(start + o_seg) * H + h) * D + ch * 8;
          valid = true;
        } else if (o_seg < 0 && hist != nullptr) {
          src = hist + ((static_cast<int64_t>(j * (KW - 1) + (KW - 1) + o_seg) * 3 + st) * H + h) * D + ch * 8;
          valid = true;
        }
        cp_async16(&raw_st[(st * HR + r) * D + ch * 8], src, valid);
      }
    }
    if (tid < 2 * C) {
      const int u = tid & (C - 1);
      const int o_seg = c0n + u;
      const bool valid = o_seg < len;
      const float* src = (tid < C ? p.alpha : p.eta) + (static_cast<int64_t>(start + (valid ? o_seg : 0)) * H + h);
      cp_async4(tid < C ? &ga[u] : &ge[u], src, valid);
    }
    asm volatile("cp.async.commit_group;\n" ::);
  };
  // a CTA-wide bounded wait on an MMA commit barrier
  auto wait_all = [&](int b, uint32_t parity) -> bool {
    const bool ok = tc::mbar_wait(&bars[b], parity, abort);
    const bool all = __syncthreads_and(ok) != 0;
    tc::tc_fence_after();
    return all;
  };

  // ---- initial state into TMEM (row = v, this thread's 64 columns) ------------
  {
    uint32_t v32[32];
    for (int q = 0; q < 2; ++q) {
      const int c0 = half * 64 + q * 32;
#pragma unroll
      for (int e = 0; e < 32; ++e)
        v32[e] = S0 ? __float_as_uint(S0[state_base + static_cast<int64_t>(row) * D + c0 + e]) : 0u;
      tc::tmem_st32(tmem + TS + lane_base + c0, v32);
    }
    tc::tmem_wait_st();
  }
  if (!BRANCH && ck >= 0 && ck - pos0 == 0 && p.S_ckpt && S0) {
    for (int e = tid; e < D * D; e += NT) p.S_ckpt[state_base + e] = S0[state_base + e];
  } else if (!BRANCH && ck >= 0 && ck - pos0 == 0 && p.S_ckpt) {
    for (int e = tid; e < D * D; e += NT) p.S_ckpt[state_base + e] = 0.f;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();

  unsigned char* ktg = sm + Lay::AM;  // 128 x 64 fp32 (2 boxes), over the inverse's buffers
  const uint32_t xqk_a = smem_u32(xqk), tb_a = smem_u32(tb), pb_a = smem_u32(pb), ktg_a = smem_u32(ktg);
  for (int e = tid; e < C * C; e += NT) {  // blocks of T above the diagonal stay zero
    const int t = e >> 6, sidx = e & 63;
    if ((sidx >> 4) > (t >> 4)) *reinterpret_cast<uint32_t*>(tb + swz(64, t, sidx)) = 0u;
  }
  bool ok = true;
  if (len > 0) prefetch(0);
  int ci = 0;
  for (int c0 = 0; ok && c0 < len; c0 += C, ++ci) {
    const int n = min(C, len - c0);
    const bool need_state = !BRANCH || (c0 + C < len);
    const uint32_t par = static_cast<uint32_t>(ci & 1);
    asm volatile("cp.async.wait_group 0;\n" ::);
    __syncthreads();
    // ---- gates (warp 0) --------------------------------------------------------
    if (warp == 0) {
      const int u0 = 2 * lane, u1 = u0 + 1;
      const float l0 = u0 < n ? logf(ga[u0]) : 0.f, l1 = u1 < n ? logf(ga[u1]) : 0.f;
      float x = l0 + l1;
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const float g1 = x, g0 = x - l1;
      const float glast = __shfl_sync(0xffffffffu, x, 31);
      G[u0] = g0;
      G[u1] = g1;
      EG[u0] = expf(g0);
      EG[u1] = expf(g1);
      GL[u0] = expf(glast - g0);
      GL[u1] = expf(glast - g1);
      ETA[u0] = u0 < n ? ge[u0] : 0.f;
      ETA[u1] = u1 < n ? ge[u1] : 0.f;
    }
    // ---- conv + SiLU: thread = (channel c, half of the rows), the three streams
    //      interleaved; q, k into the swizzled [Q; K] tile, v into the plain tile ----
    {
      const int c = tid >> 1, u0 = (tid & 1) * 32;
      float w[3][KW], x0[3], x1[3], x2[3];
      const uint16_t* col[3];
#pragma unroll
      for (int st = 0; st < 3; ++st) {
        const float* wp = p.conv_w + ((static_cast<int64_t>(st) * H + h) * D + c) * KW;
#pragma unroll
        for (int i = 0; i < KW; ++i) w[st][i] = wp[i];
        col[st] = &raw_st[st * HR * D + c];
        x0[st] = bf2f(col[st][u0 * D]);
        x1[st] = bf2f(col[st][(u0 + 1) * D]);
        x2[st] = bf2f(col[st][(u0 + 2) * D]);
      }
#pragma unroll 2
      for (int u = u0; u < u0 + 32; ++u) {
        float y[3];
#pragma unroll
        for (int st = 0; st < 3; ++st) {
          const float x3 = bf2f(col[st][(u + 3) * D]);
          y[st] = u < n ? silu(w[st][0] * x0[st] + w[st][1] * x1[st] + w[st][2] * x2[st] + w[st][3] * x3) : 0.f;
          x0[st] = x1[st];
          x1[st] = x2[st];
          x2[st] = x3;
        }
        *reinterpret_cast<float*>(xqk + swz(128, u, c)) = y[0];
        *reinterpret_cast<float*>(xqk + swz(128, C + u, c)) = y[1];
        vh[u * LDV + c] = y[2];
      }
    }
    __syncthreads();
    if (c0 + C < len) prefetch(c0 + C);
    // ---- L2 normalisation of the 128 q/k rows (4 rows in flight per warp), TF32 ----
    for (int r0 = warp * 4; r0 < 2 * C; r0 += 4 * (NT / 32)) {
      float x[4][4], ss[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        ss[q] = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[q][k] = *reinterpret_cast<const float*>(xqk + swz(128, r0 + q, lane + 32 * k));
          ss[q] += x[q][k] * x[q][k];
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int q = 0; q < 4; ++q) ss[q] += __shfl_xor_sync(0xffffffffu, ss[q], o);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float inv = rsqrtf_(ss[q] + 1e-6f);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint32_t*>(xqk + swz(128, r0 + q, lane + 32 * k)) = tf32_bits(x[q][k] * inv);
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    // ---- M1 and M3 ----------------------------------------------------------------
    if (tid == 0) {
      tc::tc_fence_after();
      constexpr uint32_t id1 = tc::idesc_tf32(128, 64, 0, 0);
      constexpr uint32_t id3 = tc::idesc_tf32(128, 128, 0, 0);
      // the start-address field is in 16-byte units: +2 per 32-byte k step, +1024 per box
      const uint64_t dq = tc::sdesc_sw128(xqk_a, 16, 1024), dk = tc::sdesc_sw128(xqk_a + C * 128, 16, 1024);
#pragma unroll
      for (int ks = 0; ks < D / 8; ++ks) {
        const uint64_t off = static_cast<uint64_t>((ks >> 2) * 1024 + (ks & 3) * 2);
        tc::mma_tf32_ss(tmem + TD1, dq + off, dk + off, id1, ks > 0);
      }
      tc::mma_commit(&bars[B_M1]);
#pragma unroll
      for (int ks = 0; ks < D / 8; ++ks) {
        const uint64_t off = static_cast<uint64_t>((ks >> 2) * 1024 + (ks & 3) * 2);
        tc::mma_tf32_ts(tmem + TD3, tmem + TS + ks * 8, dq + off, id3, ks > 0);
      }
      tc::mma_commit(&bars[B_M3]);
    }
    if (!(ok = wait_all(B_M1, par))) break;
    // ---- P (q rows) and A (k rows) from [Q; K] K^T --------------------------------
    {
      uint32_t v32[32];
      tc::tmem_ld32(tmem + TD1 + lane_base + half * 32, v32);
      tc::tmem_wait_ld();
      const int t = row < C ? row : row - C;
      const float gt = G[t] * kLog2e, et = ETA[t];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int s = half * 32 + e;
        const float gam = s <= t ? ex2f(gt - G[s] * kLog2e) : 0.f;
        const float val = __uint_as_float(v32[e]);
        if (row < C) *reinterpret_cast<uint32_t*>(pb + swz(64, t, s)) = tf32_bits(gam * val);
        else am[t * LDC + s] = s < t ? et * gam * val : 0.f;
      }
    }
    __syncthreads();
    // ---- T = (I + A)^{-1} (fp32): diagonal 16x16 blocks, then the others; each
    //      finished block also goes (rounded) into the B-operand tile -------------
    if (tid < 64) {
      const int bi = tid >> 4, c = tid & 15, base = bi * 16;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float a0 = (r == c) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
        for (int m = 0; m < r; m += 2) {
          a0 -= am[(base + r) * LDC + base + m] * x[m];
          if (m + 1 < r) a1 -= am[(base + r) * LDC + base + m + 1] * x[m + 1];
        }
        x[r] = r < c ? 0.f : a0 + a1;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        tm[(base + r) * LDC + base + c] = x[r];
        *reinterpret_cast<uint32_t*>(tb + swz(64, base + r, base + c)) = tf32_bits(x[r]);
      }
    }
    __syncthreads();
    for (int dist = 1; dist < 4; ++dist) {
      const int npair = 4 - dist;
      for (int e = tid; e < npair * 256; e += NT) {
        const int pr = e >> 8, r = (e >> 4) & 15, c = e & 15;
        const int bi = dist + pr, bj = pr;
        const float* arow = am + (bi * 16 + r) * LDC;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        for (int m = bj * 16; m < bi * 16; m += 4) {
          a0 += arow[m] * tm[m * LDC + bj * 16 + c];
          a1 += arow[m + 1] * tm[(m + 1) * LDC + bj * 16 + c];
          a2 += arow[m + 2] * tm[(m + 2) * LDC + bj * 16 + c];
          a3 += arow[m + 3] * tm[(m + 3) * LDC + bj * 16 + c];
        }
        xs[e] = (a0 + a1) + (a2 + a3);
      }
      __syncthreads();
      for (int e = tid; e < npair * 256; e += NT) {
        const int pr = e >> 8, r = (e >> 4) & 15, c = e & 15;
        const int bi = dist + pr, bj = pr;
        const float* trow = tm + (bi * 16 + r) * LDC + bi * 16;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
          a0 += trow[m] * xs[(pr << 8) + m * 16 + c];
          a1 += trow[m + 1] * xs[(pr << 8) + (m + 1) * 16 + c];
          a2 += trow[m + 2] * xs[(pr << 8) + (m + 2) * 16 + c];
          a3 += trow[m + 3] * xs[(pr << 8) + (m + 3) * 16 + c];
        }
        const float v = -((a0 + a1) + (a2 + a3));
        tm[(bi * 16 + r) * LDC + bj * 16 + c] = v;
        *reinterpret_cast<uint32_t*>(tb + swz(64, bi * 16 + r, bj * 16 + c)) = tf32_bits(v);
      }
      __syncthreads();
    }
    // the inverse's buffers are free from here on (the last loop ended with a barrier)
    // K^T diag(Gamma_last) as the B operand of the state update (row c, column s),
    // written over the inverse's buffers
    if (need_state) {
      const int cch = tid >> 1, s0 = (tid & 1) * 32;
#pragma unroll 8
      for (int sidx = s0; sidx < s0 + 32; ++sidx) {
        const float kv = *reinterpret_cast<const float*>(xqk + swz(128, C + sidx, cch));
        *reinterpret_cast<uint32_t*>(ktg + swz(128, cch, sidx)) = tf32_bits(GL[sidx] * kv);
      }
    }
    tc::fence_proxy_async_smem();
    if (!(ok = wait_all(B_M3, par))) break;
    // ---- from S [Q; K]^T: O^T starts at e^G (Q S^T)^T, R^T = eta (V - e^G K S^T)^T ----
    {
      uint32_t v32[32];
      for (int q = 0; q < 2; ++q) {
        const int tc0 = q * 32;
        const uint32_t col = TD3 + half * 64 + tc0;  // half 0: q tokens, half 1: k tokens
        tc::tmem_ld32(tmem + col + lane_base, v32);
        tc::tmem_wait_ld();
        if (half == 0) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v32[e] = __float_as_uint(__uint_as_float(v32[e]) * EG[tc0 + e]);
          tc::tmem_st32(tmem + col + lane_base, v32);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int t = tc0 + e;
            v32[e] = tf32_bits(ETA[t] * (vh[t * LDV + row] - EG[t] * __uint_as_float(v32[e])));
          }
          tc::tmem_st32(tmem + TR + tc0 + lane_base, v32);
        }
      }
      tc::tmem_wait_st();
    }
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc::tc_fence_after();
      constexpr uint32_t id4 = tc::idesc_tf32(128, 64, 0, 0);
      for (int ks = 0; ks < C / 8; ++ks)
        tc::mma_tf32_ts(tmem + TU, tmem + TR + ks * 8,
                        tc::sdesc_sw128(tb_a + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), id4, ks > 0);
      tc::mma_commit(&bars[B_M4]);
    }
    if (!(ok = wait_all(B_M4, par))) break;
    // ---- U^T rounded to TF32 in place (A operand of M5 and M6) ---------------------
    {
      uint32_t v32[32];
      tc::tmem_ld32(tmem + TU + half * 32 + lane_base, v32);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) v32[e] = tf32_bits(__uint_as_float(v32[e]));
      tc::tmem_st32(tmem + TU + half * 32 + lane_base, v32);
      tc::tmem_wait_st();
    }
    // ---- checkpoint inside this chunk (rare): state after r_ck of its tokens -------
    if (!BRANCH && ck >= 0 && p.S_ckpt) {
      const int r_ck = ck - pos0 - c0;
      if (r_ck >= 1 && r_ck <= n) {
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
        if (half == 0) {
          uint32_t u32a[32], u32b[32], s32[32];
          tc::tmem_ld32(tmem + TU + lane_base, u32a);
          tc::tmem_ld32(tmem + TU + 32 + lane_base, u32b);
          tc::tmem_wait_ld();
          const float gr = G[r_ck - 1];
          for (int cb = 0; cb < D; cb += 32) {
            tc::tmem_ld32(tmem + TS + cb + lane_base, s32);
            tc::tmem_wait_ld();
            float acc[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[e] = expf(gr) * __uint_as_float(s32[e]);
            for (int s = 0; s < r_ck; ++s) {
              const float us = __uint_as_float(s < 32 ? u32a[s & 31] : u32b[s & 31]) * expf(gr - G[s]);
#pragma unroll
              for (int e = 0; e < 32; ++e) acc[e] += us * *reinterpret_cast<const float*>(xqk + swz(128, C + s, cb + e));
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) p.S_ckpt[state_base + static_cast<int64_t>(row) * D + cb + e] = acc[e];
          }
        }
      }
    }
    // ---- S <- e^{G_last} S before the update is accumulated on it -----------------
    if (need_state) {
      const float egl = EG[C - 1];
      uint32_t v32[32];
      for (int q = 0; q < 2; ++q) {
        const uint32_t col = TS + half * 64 + q * 32;
        tc::tmem_ld32(tmem + col + lane_base, v32);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) v32[e] = __float_as_uint(__uint_as_float(v32[e]) * egl);
        tc::tmem_st32(tmem + col + lane_base, v32);
      }
      tc::tmem_wait_st();
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc::tc_fence_after();
      constexpr uint32_t id5 = tc::idesc_tf32(128, 64, 0, 0);
      constexpr uint32_t id6 = tc::idesc_tf32(128, 128, 0, 0);
      for (int ks = 0; ks < C / 8; ++ks)
        tc::mma_tf32_ts(tmem + TD3, tmem + TU + ks * 8,
                        tc::sdesc_sw128(pb_a + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), id5, 1u);
      if (need_state)
        for (int ks = 0; ks < C / 8; ++ks)
          tc::mma_tf32_ts(tmem + TS, tmem + TU + ks * 8,
                          tc::sdesc_sw128(ktg_a + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024), id6, 1u);
      tc::mma_commit(&bars[B_M56]);
    }
    if (!(ok = wait_all(B_M56, par))) break;
    // ---- O^T (lane v, token columns) -> bf16 rows of the output ----------------------
    {
      uint16_t* ost = reinterpret_cast<uint16_t*>(vh);  // [C][D + 8] bf16 (v is no longer needed)
      constexpr int LDO = D + 8;
      uint32_t v32[32];
      tc::tmem_ld32(tmem + TD3 + half * 32 + lane_base, v32);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) ost[(half * 32 + e) * LDO + row] = f2bf(__uint_as_float(v32[e]));
      __syncthreads();
      constexpr int CPR = D / 8;
      for (int e = tid; e < n * CPR; e += NT) {
        const int t = e / CPR, ch = e % CPR;
        *reinterpret_cast<uint4*>(p.o + (static_cast<int64_t>(start + c0 + t) * H + h) * D + ch * 8) =
            *reinterpret_cast<const uint4*>(&ost[t * LDO + ch * 8]);
      }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
  }

  if (ok && !BRANCH) {
    // S_P from TMEM; conv windows from the raw rows
    uint32_t v32[32];
    for (int q = 0; q < 2; ++q) {
      const int c0 = half * 64 + q * 32;
      tc::tmem_ld32(tmem + TS + c0 + lane_base, v32);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) p.S_P[state_base + static_cast<int64_t>(row) * D + c0 + e] = __uint_as_float(v32[e]);
    }
    for (int e = tid; e < (KW - 1) * 3 * D; e += NT) {
      const int i = e / (3 * D), s = (e / D) % 3, c = e % D;
      const int64_t dst = ((static_cast<int64_t>(j * (KW - 1) + i) * 3 + s) * H + h) * D + c;
      p.conv_win[dst] = f2bf(raw(len - (KW - 1) + i, s, c));
      if (ck >= 0 && p.conv_ckpt) p.conv_ckpt[dst] = f2bf(raw(ck - pos0 - (KW - 1) + i, s, c));
    }
  }
  // every MMA issued has completed (the last wait covered them; on abort, drain)
  if (tid == 0) {
    tc::mma_commit(&bars[B_FIN]);
    tc::mbar_wait(&bars[B_FIN], 0, abort);
  }
  asm volatile("cp.async.wait_group 0;\n" ::);
  tc::tc_fence_before();
  __syncthreads();
  if (*abort && tid == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_TIMEOUT);
  if (warp == 0) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

int launch_gdn_tc(const GdnParams& p, bool branch, int grid_x, cudaStream_t s) {
  dim3 grid(grid_x, p.H);
  if (branch) {
    if (cudaFuncSetAttribute(gdn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM) !=
        cudaSuccess)
      return FORK_ECUDA;
    gdn_tc_kernel<true><<<grid, NT, Lay::SMEM, s>>>(p);
  } else {
    if (cudaFuncSetAttribute(gdn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM) !=
        cudaSuccess)
      return FORK_ECUDA;
    gdn_tc_kernel<false><<<grid, NT, Lay::SMEM, s>>>(p);
  }
  return cuda_rc(cudaGetLastError());
}

}  // namespace fork
