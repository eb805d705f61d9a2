// Two-call forked Gated DeltaNet over the flat stream.
//
// Recurrence (rainbus summary "前置知识"): per head, after a short causal conv
// (+SiLU) on q, k, v and an L2 normalisation of q and k,
//     S_t = alpha_t S_{t-1} (I - eta_t k_t k_t^T) + eta_t v_t k_t^T,   o_t = S_t q_t.
// Two calls (onedev summary "무엇과 다른가"; rainbus "方法步骤详情" step 2): call 1
// runs every trunk segment from zero (or from a resumed checkpoint) and writes
// each request's float32 S_P and conv window; call 2 runs every question
// segment at once, each starting from S_P[j] and the trunk's conv window by
// index (no state copy).
//
// Chunk form (the chunked linear-recurrence solve the DFlash-TfM summary
// describes for GDN, "GDN을 위한 롤백 없는 트리 검증": Gram matrix, masked
// triangular solve (I + X) U = beta V, output): with the chunk's start state
// S0, G_t = sum_{s<=t} log alpha_s and Gamma_ts = exp(G_t - G_s),
//   u_t = eta_t (v_t - alpha_t S_{t-1} k_t),  S_t = alpha_t S_{t-1} + u_t k_t^T,
//   (I + A) U = diag(eta) (V - diag(e^G) K S0^T),  A_ts = eta_t Gamma_ts k_t.k_s (s<t),
//   O = diag(e^G) Q S0^T + (tril(Gamma) * Q K^T) U,
//   S_end = e^{G_last} S0 + U^T diag(Gamma_last,.) K.
// One CTA per (segment, head) keeps S (d x d, float32) in shared memory for
// the whole segment.  The contractions run on the tensor cores with TF32
// operands rounded to nearest (mma.sync m16n8k8), accumulation in float32;
// T = (I + A)^{-1} is formed by blocked forward substitution in float32.
// Chunks are aligned to the segment start, so a question's result never
// depends on the rest of the round.
#include "fork_gdn.cuh"

namespace fork {



namespace {
constexpr int C = 64;         // chunk length
constexpr int NT = 256;       // threads (8 warps)
constexpr int LDC = C + 8;    // stride of 64-wide fp32 tiles (== 8 mod 32)
constexpr int KW = 4;         // conv width
constexpr int HR = C + KW - 1;  // staged raw rows per chunk (history + chunk)

template <int D>
struct GdnSmem {
  static constexpr int LDD = D + 8;  // stride of D-wide fp32 tiles (== 8 mod 32)
  float Qh[C * LDD];   // normalised q of the chunk; later the bf16 output staging
  float Kh[C * LDD];   // normalised k
  float Vh[C * LDD];   // conv'd v
  float Pm[C * LDC];   // tril(Gamma) * Q K^T
  float Am[C * LDC];   // strictly lower eta Gamma K K^T
  float Tm[C * LDC];   // (I + A)^{-1}
  float X[3 * 256];    // scratch of the blocked inverse
  uint16_t raw[3 * HR * D];  // staged raw q, k, v rows (bf16) of the next chunk
  float ga[C], ge[C];  // staged alpha, eta of the next chunk
  float G[C];          // inclusive cumulative log alpha
  float EG[C];         // exp(G)
  float GL[C];         // exp(G_last - G_s)
  float ETA[C];
};

__device__ __forceinline__ uint32_t tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void mma_tf32(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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

// Every contraction below sums over an index k in blocks of 8.  Inside a
// block the fragment slot k' = t (t = lane % 4) carries index 2t and slot
// k' = t + 4 carries 2t + 1 (the same on both operands, so the sum is
// unchanged).  This makes an accumulator tile (columns 2t, 2t+1 per thread)
// directly usable as the A operand of the next product, and turns shared
// memory operand loads into float2 loads.
struct Frag {
  uint32_t a0, a1, a2, a3;
};
// A operand from an accumulator tile acc[4] = {(g,2t), (g,2t+1), (g+8,2t), (g+8,2t+1)}.
__device__ __forceinline__ Frag a_from_acc(const float* acc) {
  return {tf32(acc[0]), tf32(acc[2]), tf32(acc[1]), tf32(acc[3])};
}
// A operand rows m0.., block k0, from a row-major fp32 tile.
__device__ __forceinline__ Frag a_from_rows(const float* base, int ld, int m0, int k0, int g, int t) {
  const float2 lo = *reinterpret_cast<const float2*>(base + (m0 + g) * ld + k0 + 2 * t);
  const float2 hi = *reinterpret_cast<const float2*>(base + (m0 + g + 8) * ld + k0 + 2 * t);
  return {tf32(lo.x), tf32(hi.x), tf32(lo.y), tf32(hi.y)};
}
// B operand B[k][n] = X[n][k] (X row-major), tile (k0, n0).
__device__ __forceinline__ void b_from_rows(const float* base, int ld, int k0, int n0, int g, int t,
                                            uint32_t& b0, uint32_t& b1) {
  const float2 v = *reinterpret_cast<const float2*>(base + (n0 + g) * ld + k0 + 2 * t);
  b0 = tf32(v.x);
  b1 = tf32(v.y);
}
__device__ __forceinline__ void mma(float* c, const Frag& a, uint32_t b0, uint32_t b1) {
  mma_tf32(c, a.a0, a.a1, a.a2, a.a3, b0, b1);
}
}  // namespace

// One CTA per (segment, head).  The state S (d x d, rows = v index) lives in
// registers: warp w < d/16 holds rows 16w..16w+15 as an accumulator tile.
// Per chunk (all products TF32 on the tensor cores, float32 accumulation):
//   M1  [Q; K] K^T            -> P = tril(Gamma) * QK^T, A = eta Gamma KK^T (strict)
//   T = (I + A)^{-1}          (float32, blocked forward substitution)
//   M3  S [K; Q]^T            -> (K S^T)^T, (Q S^T)^T               (A = S from registers)
//   R^T = eta (V - e^G K S^T)^T;  U^T = R^T T^T;  O^T = e^G (Q S^T)^T + U^T P^T
//   S  <- e^{G_last} S + U^T diag(Gamma_last) K
template <int D, bool BRANCH>
__global__ void __launch_bounds__(NT, 1) gdn_chunk_kernel(const GdnParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  GdnSmem<D>& sm = *reinterpret_cast<GdnSmem<D>*>(smem_raw);
  constexpr int LDD = GdnSmem<D>::LDD;
  constexpr int NTD = D / 8;    // 8-wide tiles over d
  constexpr int NWS = D / 16;   // warps holding the state
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
  if (p.checks && !gdn_segs_in_bounds(meta, L, seg, seg + 1, j)) {
    if (threadIdx.x == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_CHECK);
    return;
  }
  const int h = blockIdx.y;
  const int H = p.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
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
  // history rows (raw inputs before the segment): trunk -> resume window or zeros;
  // question -> its request's trunk window, by index
  const uint16_t* hist = (BRANCH || resumed) ? p.hist_in : nullptr;
  const float* S0 = (BRANCH || resumed) ? p.state_in : nullptr;
  const int64_t state_base = (static_cast<int64_t>(j) * H + h) * D * D;
  const uint16_t* xs[3] = {p.q, p.k, p.v};

  auto raw = [&](int o_seg, int s, int c) -> float {
    if (o_seg >= 0) return bf2f(xs[s][(static_cast<int64_t>(start + o_seg) * H + h) * D + c]);
    const int r = KW - 1 + o_seg;
    if (r < 0 || hist == nullptr) return 0.f;
    return bf2f(hist[((static_cast<int64_t>(j * (KW - 1) + r) * 3 + s) * H + h) * D + c]);
  };
  // stage raw rows c0n-3 .. c0n+C-1 (zero beyond the segment) and the gates of a chunk
  auto prefetch = [&](int c0n) {
    constexpr int CPR = D / 8;
    for (int e = tid; e < 3 * HR * CPR; e += NT) {
      const int s = e / (HR * CPR), r = (e / CPR) % HR, ch = e % CPR;
      const int o_seg = c0n - (KW - 1) + r;
      const uint16_t* src = p.q;
      bool valid = false;
      if (o_seg >= 0 && o_seg < len) {
        src = xs[s] + (static_cast<int64_t>(start + o_seg) * H + h) * D + ch * 8;
        valid = true;
      } else if (o_seg < 0 && hist != nullptr) {
        src = hist + ((static_cast<int64_t>(j * (KW - 1) + (KW - 1) + o_seg) * 3 + s) * H + h) * D + ch * 8;
        valid = true;
      }
      cp_async16(&sm.raw[(s * HR + r) * D + ch * 8], src, valid);
    }
    for (int u = tid; u < 2 * C; u += NT) {
      const int o_seg = c0n + (u % C);
      const bool valid = o_seg < len;
      const float* src = (u < C ? p.alpha : p.eta) + (static_cast<int64_t>(start + (valid ? o_seg : 0)) * H + h);
      cp_async4(u < C ? &sm.ga[u] : &sm.ge[u - C], src, valid);
    }
    asm volatile("cp.async.commit_group;\n" ::);
  };

  // state rows of this warp, as an accumulator tile
  float st[NTD][4];
  const bool holds_state = warp < NWS;
  const int m0 = warp * 16;  // first state row of this warp
#pragma unroll
  for (int nt = 0; nt < NTD; ++nt) {
    st[nt][0] = st[nt][1] = st[nt][2] = st[nt][3] = 0.f;
    if (holds_state && S0) {
      const int cc = nt * 8 + 2 * t4;
      const float2 a = *reinterpret_cast<const float2*>(S0 + state_base + (m0 + g) * D + cc);
      const float2 b = *reinterpret_cast<const float2*>(S0 + state_base + (m0 + g + 8) * D + cc);
      st[nt][0] = a.x;
      st[nt][1] = a.y;
      st[nt][2] = b.x;
      st[nt][3] = b.y;
    }
  }
  auto store_state = [&](float* dst, const float (*v)[4]) {
#pragma unroll
    for (int nt = 0; nt < NTD; ++nt) {
      const int cc = nt * 8 + 2 * t4;
      *reinterpret_cast<float2*>(dst + state_base + (m0 + g) * D + cc) = make_float2(v[nt][0], v[nt][1]);
      *reinterpret_cast<float2*>(dst + state_base + (m0 + g + 8) * D + cc) = make_float2(v[nt][2], v[nt][3]);
    }
  };
  if (!BRANCH && ck >= 0 && ck - pos0 == 0 && p.S_ckpt && holds_state) store_state(p.S_ckpt, st);

  if (len > 0) prefetch(0);
  for (int c0 = 0; c0 < len; c0 += C) {
    const int n = min(C, len - c0);
    const bool need_state = !BRANCH || (c0 + C < len);
    asm volatile("cp.async.wait_group 0;\n" ::);
    __syncthreads();
    // ---- gates (warp 0): G = inclusive cumsum of log alpha ---------------------
    if (warp == 0) {
      const int u0 = 2 * lane, u1 = u0 + 1;
      const float l0 = u0 < n ? logf(sm.ga[u0]) : 0.f, l1 = u1 < n ? logf(sm.ga[u1]) : 0.f;
      float x = l0 + l1;
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const float g1 = x, g0 = x - l1;
      const float glast = __shfl_sync(0xffffffffu, x, 31);
      sm.G[u0] = g0;
      sm.G[u1] = g1;
      sm.EG[u0] = expf(g0);
      sm.EG[u1] = expf(g1);
      sm.GL[u0] = expf(glast - g0);
      sm.GL[u1] = expf(glast - g1);
      sm.ETA[u0] = u0 < n ? sm.ge[u0] : 0.f;
      sm.ETA[u1] = u1 < n ? sm.ge[u1] : 0.f;
    }
    // ---- conv + SiLU from the staged rows: item = (stream, channel, half) -------
    for (int it = tid; it < 3 * D * 2; it += NT) {
      const int s = it / (2 * D), c = (it / 2) % D, hf = it % 2;
      const float* w = p.conv_w + ((static_cast<int64_t>(s) * H + h) * D + c) * KW;
      const float w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3];
      const uint16_t* col = &sm.raw[s * HR * D + c];
      float* dst = s == 0 ? sm.Qh : (s == 1 ? sm.Kh : sm.Vh);
      const int u0 = hf * 32;
      float x0 = bf2f(col[u0 * D]), x1 = bf2f(col[(u0 + 1) * D]), x2 = bf2f(col[(u0 + 2) * D]);
#pragma unroll 4
      for (int u = u0; u < u0 + 32; ++u) {
        const float x3 = bf2f(col[(u + 3) * D]);
        float y = w0 * x0 + w1 * x1 + w2 * x2 + w3 * x3;
        y = y / (1.f + expf(-y));
        dst[u * LDD + c] = u < n ? y : 0.f;
        x0 = x1;
        x1 = x2;
        x2 = x3;
      }
    }
    __syncthreads();
    if (c0 + C < len) prefetch(c0 + C);  // the staging buffer is free again
    // ---- L2 normalisation of q and k rows --------------------------------------
    for (int u = warp; u < 2 * C; u += NT / 32) {
      float* row = (u < C) ? &sm.Qh[u * LDD] : &sm.Kh[(u - C) * LDD];
      float ss = 0.f;
      for (int c = lane; c < D; c += 32) ss += row[c] * row[c];
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float inv = 1.f / sqrtf(ss + 1e-6f);
      for (int c = lane; c < D; c += 32) row[c] *= inv;
    }
    __syncthreads();

    // ---- M1: [Q; K] K^T -> P (warps 0-3) and A (warps 4-7) -----------------------
    {
      const float* Xs = warp < 4 ? sm.Qh : sm.Kh;
      const int r0 = (warp & 3) * 16;
      float acc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll 2
      for (int k0 = 0; k0 < D; k0 += 8) {
        const Frag a = a_from_rows(Xs, LDD, r0, k0, g, t4);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          uint32_t b0, b1;
          b_from_rows(sm.Kh, LDD, k0, nt * 8, g, t4, b0, b1);
          mma(acc[nt], a, b0, b1);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int tr = r0 + g + hh * 8;
          const int sc = nt * 8 + 2 * t4;
          const float v0 = acc[nt][2 * hh], v1 = acc[nt][2 * hh + 1];
          const float gam0 = sc <= tr ? expf(sm.G[tr] - sm.G[sc]) : 0.f;
          const float gam1 = sc + 1 <= tr ? expf(sm.G[tr] - sm.G[sc + 1]) : 0.f;
          if (warp < 4) {
            *reinterpret_cast<float2*>(&sm.Pm[tr * LDC + sc]) = make_float2(gam0 * v0, gam1 * v1);
          } else {
            const float et = sm.ETA[tr];
            *reinterpret_cast<float2*>(&sm.Am[tr * LDC + sc]) =
                make_float2(sc < tr ? et * gam0 * v0 : 0.f, sc + 1 < tr ? et * gam1 * v1 : 0.f);
          }
        }
      }
    }
    __syncthreads();
    // ---- T = (I + A)^{-1}: diagonal 16x16 blocks, then off-diagonal blocks -------
    if (tid < 64) {
      const int bi = tid >> 4, c = tid & 15, base = bi * 16;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < r; ++m) acc -= sm.Am[(base + r) * LDC + base + m] * x[m];
        x[r] = r < c ? 0.f : acc;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) sm.Tm[(base + r) * LDC + base + c] = x[r];
    }
    __syncthreads();
    for (int dist = 1; dist < 4; ++dist) {
      const int npair = 4 - dist;
      for (int e = tid; e < npair * 256; e += NT) {
        const int pr = e >> 8, r = (e >> 4) & 15, c = e & 15;
        const int bi = dist + pr, bj = pr;
        float acc = 0.f;
        for (int m = bj * 16; m < bi * 16; ++m) acc += sm.Am[(bi * 16 + r) * LDC + m] * sm.Tm[m * LDC + bj * 16 + c];
        sm.X[e] = acc;
      }
      __syncthreads();
      for (int e = tid; e < npair * 256; e += NT) {
        const int pr = e >> 8, r = (e >> 4) & 15, c = e & 15;
        const int bi = dist + pr, bj = pr;
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) acc += sm.Tm[(bi * 16 + r) * LDC + bi * 16 + m] * sm.X[(pr << 8) + m * 16 + c];
        sm.Tm[(bi * 16 + r) * LDC + bj * 16 + c] = -acc;
      }
      __syncthreads();
    }

    // ---- state products (warps holding S) ---------------------------------------
    float rk[8][4];  // (K S^T)^T, then R^T
    float oq[8][4];  // e^G (Q S^T)^T, then O^T
    float ut[8][4];  // U^T
    if (holds_state) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        rk[i][0] = rk[i][1] = rk[i][2] = rk[i][3] = oq[i][0] = oq[i][1] = oq[i][2] = oq[i][3] = 0.f;
#pragma unroll
      for (int kb = 0; kb < NTD; ++kb) {
        const Frag a = a_from_acc(st[kb]);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          uint32_t b0, b1;
          b_from_rows(sm.Kh, LDD, kb * 8, nt * 8, g, t4, b0, b1);
          mma(rk[nt], a, b0, b1);
          b_from_rows(sm.Qh, LDD, kb * 8, nt * 8, g, t4, b0, b1);
          mma(oq[nt], a, b0, b1);
        }
      }
      // R^T[v][t] = eta_t (V[t][v] - e^{G_t} (K S^T)^T[v][t]);  O^T starts at e^{G_t} (Q S^T)^T
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = m0 + g + (e >> 1) * 8, t = nt * 8 + 2 * t4 + (e & 1);
          const float eg = sm.EG[t];
          rk[nt][e] = sm.ETA[t] * (sm.Vh[t * LDD + v] - eg * rk[nt][e]);
          oq[nt][e] *= eg;
        }
      }
      // U^T = R^T T^T   (T lower triangular: block kb contributes to token tiles nt >= kb)
#pragma unroll
      for (int i = 0; i < 8; ++i) ut[i][0] = ut[i][1] = ut[i][2] = ut[i][3] = 0.f;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        const Frag a = a_from_acc(rk[kb]);
#pragma unroll
        for (int nt = kb; nt < 8; ++nt) {
          uint32_t b0, b1;
          b_from_rows(sm.Tm, LDC, kb * 8, nt * 8, g, t4, b0, b1);
          mma(ut[nt], a, b0, b1);
        }
      }
      // O^T += U^T P^T   (P lower triangular incl. diagonal)
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        const Frag a = a_from_acc(ut[kb]);
#pragma unroll
        for (int nt = kb; nt < 8; ++nt) {
          uint32_t b0, b1;
          b_from_rows(sm.Pm, LDC, kb * 8, nt * 8, g, t4, b0, b1);
          mma(oq[nt], a, b0, b1);
        }
      }
    }
    __syncthreads();  // every warp is done reading Qh: reuse it to stage the output
    uint16_t* ost = reinterpret_cast<uint16_t*>(sm.Qh);  // [C][D + 8] bf16
    constexpr int LDO = D + 8;
    if (holds_state) {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = m0 + g + (e >> 1) * 8, t = nt * 8 + 2 * t4 + (e & 1);
          ost[t * LDO + v] = f2bf(oq[nt][e]);
        }
      }
    }
    __syncthreads();
    {
      constexpr int CPR = D / 8;
      for (int e = tid; e < n * CPR; e += NT) {
        const int t = e / CPR, ch = e % CPR;
        *reinterpret_cast<uint4*>(p.o + (static_cast<int64_t>(start + c0 + t) * H + h) * D + ch * 8) =
            *reinterpret_cast<const uint4*>(&ost[t * LDO + ch * 8]);
      }
    }
    // ---- checkpoint inside this chunk (rare): state after r_ck of its tokens -------
    if (!BRANCH && ck >= 0 && p.S_ckpt && holds_state) {
      const int r_ck = ck - pos0 - c0;
      if (r_ck >= 1 && r_ck <= n) {
        const float gr = sm.G[r_ck - 1];
        const float egr = expf(gr);
        float sc[NTD][4];
#pragma unroll
        for (int nt = 0; nt < NTD; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[nt][e] = egr * st[nt][e];
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          const Frag a = a_from_acc(ut[kb]);
          const int s0 = kb * 8 + 2 * t4;
          const float f0 = s0 < r_ck ? expf(gr - sm.G[s0]) : 0.f;
          const float f1 = s0 + 1 < r_ck ? expf(gr - sm.G[s0 + 1]) : 0.f;
#pragma unroll
          for (int nt = 0; nt < NTD; ++nt) {
            const uint32_t b0 = tf32(f0 * sm.Kh[s0 * LDD + nt * 8 + g]);
            const uint32_t b1 = tf32(f1 * sm.Kh[(s0 + 1) * LDD + nt * 8 + g]);
            mma(sc[nt], a, b0, b1);
          }
        }
        store_state(p.S_ckpt, sc);
      }
    }
    // ---- S <- e^{G_last} S + U^T diag(Gamma_last) K ---------------------------------
    if (need_state && holds_state) {
      const float egl = sm.EG[C - 1];
#pragma unroll
      for (int nt = 0; nt < NTD; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) st[nt][e] *= egl;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        const Frag a = a_from_acc(ut[kb]);
        const int s0 = kb * 8 + 2 * t4;
        const float f0 = sm.GL[s0], f1 = sm.GL[s0 + 1];
#pragma unroll
        for (int nt = 0; nt < NTD; ++nt) {
          const uint32_t b0 = tf32(f0 * sm.Kh[s0 * LDD + nt * 8 + g]);
          const uint32_t b1 = tf32(f1 * sm.Kh[(s0 + 1) * LDD + nt * 8 + g]);
          mma(st[nt], a, b0, b1);
        }
      }
    }
    __syncthreads();
  }

  if (!BRANCH) {
    if (holds_state) store_state(p.S_P, st);
    // conv windows: raw inputs of the last K-1 positions before the end / before m
    for (int e = tid; e < (KW - 1) * 3 * D; e += NT) {
      const int i = e / (3 * D), s = (e / D) % 3, c = e % D;
      const int64_t dst = ((static_cast<int64_t>(j * (KW - 1) + i) * 3 + s) * H + h) * D + c;
      p.conv_win[dst] = f2bf(raw(len - (KW - 1) + i, s, c));
      if (ck >= 0 && p.conv_ckpt) p.conv_ckpt[dst] = f2bf(raw(ck - pos0 - (KW - 1) + i, s, c));
    }
  }
}

template <int D, bool BRANCH>
static int launch_gdn(const GdnParams& p, int grid_x, cudaStream_t s) {
  const size_t smem = sizeof(GdnSmem<D>);
  if (cuda_rc(cudaFuncSetAttribute(gdn_chunk_kernel<D, BRANCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem))) != FORK_OK)
    return FORK_ECUDA;
  dim3 grid(grid_x, p.H);
  gdn_chunk_kernel<D, BRANCH><<<grid, NT, smem, s>>>(p);
  return cuda_rc(cudaGetLastError());
}

static int gdn_common_checks(const fork_meta* m, MetaLayout* L, const uint16_t* q, const uint16_t* k,
                             const uint16_t* v, const float* alpha, const float* eta,
                             const float* conv_w, int32_t H, int32_t d, int32_t K, int32_t chunk,
                             const uint16_t* o) {
  int rc = check_meta(m, L);
  if (rc != FORK_OK) return rc;
  if (!q || !k || !v || !alpha || !eta || !conv_w || !o) return FORK_EINVAL;
  if (H < 1 || H > 65535 || (d != 64 && d != 128) || K != 4 || chunk != C) return FORK_EINVAL;
  if (!is_aligned16(q) || !is_aligned16(k) || !is_aligned16(v) || !is_aligned16(o)) return FORK_EINVAL;
  return FORK_OK;
}

}  // namespace fork

using namespace fork;

extern "C" int fork_gdn_trunk(const fork_meta* m, const uint16_t* q, const uint16_t* k,
                              const uint16_t* v, const float* alpha, const float* eta,
                              const float* conv_w, int32_t H, int32_t d, int32_t K, int32_t chunk,
                              const float* init_state, const uint16_t* init_conv, float* S_P,
                              uint16_t* conv_win, float* S_ckpt, uint16_t* conv_ckpt, uint16_t* o,
                              uint32_t flags, void* stream) {
  MetaLayout L;
  int rc = gdn_common_checks(m, &L, q, k, v, alpha, eta, conv_w, H, d, K, chunk, o);
  if (rc != FORK_OK) return rc;
  if (!S_P || !conv_win || !is_aligned16(S_P)) return FORK_EINVAL;
  if ((S_ckpt == nullptr) != (conv_ckpt == nullptr)) return FORK_EINVAL;
  if ((init_state == nullptr) != (init_conv == nullptr)) return FORK_EINVAL;
  if (init_state && !is_aligned16(init_state)) return FORK_EINVAL;
  if ((rc = check_device()) != FORK_OK) return rc;
  GdnParams p;
  p.meta = static_cast<const int32_t*>(m->d_buf);
  p.L = L;
  p.q = q;
  p.k = k;
  p.v = v;
  p.alpha = alpha;
  p.eta = eta;
  p.conv_w = conv_w;
  p.H = H;
  p.K = K;
  p.state_in = init_state;
  p.hist_in = init_conv;
  p.S_P = S_P;
  p.conv_win = conv_win;
  p.S_ckpt = S_ckpt;
  p.conv_ckpt = conv_ckpt;
  p.o = o;
  p.seg_base = 0;
  p.n_segs = -1;
  p.checks = (flags & FORK_CHECKS) ? 1 : 0;
  p.stall = (flags & FORK_TEST_STALL) ? 1 : 0;
  p.wait_ns = wait_ns_of(m);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 128 && !(flags & FORK_WARP_MMA)) return launch_gdn_tc(p, false, m->max_req, s);
  return d == 64 ? launch_gdn<64, false>(p, m->max_req, s) : launch_gdn<128, false>(p, m->max_req, s);
}

// One level of a token forest: the nodes with state indices [first, first + count), each a
// trunk whose start state and conv window are its parent's (node_state / node_conv at the
// segment's state index), writing its own at its index.
extern "C" int fork_gdn_forest(const fork_meta* m, int32_t first, int32_t count, const uint16_t* q,
                               const uint16_t* k, const uint16_t* v, const float* alpha, const float* eta,
                               const float* conv_w, int32_t H, int32_t d, int32_t K, int32_t chunk,
                               float* node_state, uint16_t* node_conv, uint16_t* o, uint32_t flags,
                               void* stream) {
  MetaLayout L;
  int rc = gdn_common_checks(m, &L, q, k, v, alpha, eta, conv_w, H, d, K, chunk, o);
  if (rc != FORK_OK) return rc;
  if (!node_state || !node_conv || !is_aligned16(node_state) || !is_aligned16(node_conv)) return FORK_EINVAL;
  if (d != 128 || (flags & FORK_WARP_MMA)) return FORK_EINVAL;
  if (first < 0 || count < 0 || static_cast<int64_t>(first) + count > m->max_req) return FORK_EINVAL;
  if ((rc = check_device()) != FORK_OK) return rc;
  if (count == 0) return FORK_OK;
  GdnParams p;
  p.meta = static_cast<const int32_t*>(m->d_buf);
  p.L = L;
  p.q = q;
  p.k = k;
  p.v = v;
  p.alpha = alpha;
  p.eta = eta;
  p.conv_w = conv_w;
  p.H = H;
  p.K = K;
  p.state_in = node_state;
  p.hist_in = node_conv;
  p.S_P = node_state;
  p.conv_win = node_conv;
  p.S_ckpt = nullptr;
  p.conv_ckpt = nullptr;
  p.o = o;
  p.seg_base = first;
  p.n_segs = count;
  p.checks = (flags & FORK_CHECKS) ? 1 : 0;
  p.stall = (flags & FORK_TEST_STALL) ? 1 : 0;
  p.wait_ns = wait_ns_of(m);
  return launch_gdn_tc(p, false, count, static_cast<cudaStream_t>(stream));
}

extern "C" int fork_gdn_branches(const fork_meta* m, const uint16_t* q, const uint16_t* k,
                                 const uint16_t* v, const float* alpha, const float* eta,
                                 const float* conv_w, int32_t H, int32_t d, int32_t K,
                                 int32_t chunk, const float* S_P, const uint16_t* conv_win,
                                 uint16_t* o, uint32_t flags, void* stream) {
  MetaLayout L;
  int rc = gdn_common_checks(m, &L, q, k, v, alpha, eta, conv_w, H, d, K, chunk, o);
  if (rc != FORK_OK) return rc;
  if (!S_P || !conv_win || !is_aligned16(S_P)) return FORK_EINVAL;
  if ((rc = check_device()) != FORK_OK) return rc;
  if (m->max_q == 0) return FORK_OK;
  GdnParams p;
  p.meta = static_cast<const int32_t*>(m->d_buf);
  p.L = L;
  p.q = q;
  p.k = k;
  p.v = v;
  p.alpha = alpha;
  p.eta = eta;
  p.conv_w = conv_w;
  p.H = H;
  p.K = K;
  p.state_in = S_P;
  p.hist_in = conv_win;
  p.S_P = nullptr;
  p.conv_win = nullptr;
  p.S_ckpt = nullptr;
  p.conv_ckpt = nullptr;
  p.o = o;
  p.seg_base = 0;
  p.n_segs = -1;
  p.checks = (flags & FORK_CHECKS) ? 1 : 0;
  p.stall = (flags & FORK_TEST_STALL) ? 1 : 0;
  p.wait_ns = wait_ns_of(m);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 128 && !(flags & FORK_WARP_MMA)) return launch_gdn_tc(p, true, m->max_q, s);
  return d == 64 ? launch_gdn<64, true>(p, m->max_q, s) : launch_gdn<128, true>(p, m->max_q, s);
}
