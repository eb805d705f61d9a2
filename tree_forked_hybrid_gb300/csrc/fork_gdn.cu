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
//   (I + A) U = diag(eta) V - diag(eta e^G) K S0^T,  A_ts = eta_t Gamma_ts k_t.k_s (s<t),
//   O = diag(e^G) Q S0^T + (tril(Gamma) * Q K^T) U,
//   S_end = e^{G_last} S0 + U^T diag(Gamma_last,.) K.
// Rows of S (the v index) evolve independently given the keys, so each CTA
// owns a slice of 32 rows; chunks are aligned to the segment start, so a
// question's result never depends on the rest of the round.
#include "fork_common.cuh"

namespace fork {

struct GdnParams {
  const int32_t* meta;
  MetaLayout L;
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const float* alpha;
  const float* eta;
  const float* conv_w;      // [3, H, D, K]
  int H, K;
  const float* state_in;    // trunk: init_state (resume) or null; branch: S_P
  const uint16_t* hist_in;  // trunk: init_conv or null; branch: conv_win
  float* S_P;               // trunk output
  uint16_t* conv_win;       // trunk output
  float* S_ckpt;
  uint16_t* conv_ckpt;
  uint16_t* o;
};

namespace {
constexpr int C = 64;     // chunk length
constexpr int DVS = 32;   // rows of S per CTA
constexpr int NT = 256;   // threads

template <int D>
struct GdnSmem {
  static constexpr int LDD = D + 1;
  static constexpr int LDV = DVS + 1;
  static constexpr int LDC = C + 1;
  float S[DVS * LDD];
  float Q[C * LDD];
  float K[C * LDD];
  float W[C * LDD];
  float U[C * LDV];
  float A[C * LDC];
  float QK[C * LDC];
  float G[C];
  float EG[C];
  float GL[C];  // Gamma_{last, s} = exp(G_last - G_s)
  float ETA[C];
};
}  // namespace

template <int D, bool BRANCH>
__global__ void __launch_bounds__(NT, 1) gdn_chunk_kernel(const GdnParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  GdnSmem<D>& sm = *reinterpret_cast<GdnSmem<D>*>(smem_raw);
  constexpr int LDD = GdnSmem<D>::LDD, LDV = GdnSmem<D>::LDV, LDC = GdnSmem<D>::LDC;
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
  const int z = blockIdx.z;  // slice of S rows [z*DVS, z*DVS + DVS)
  const int H = p.H, K = p.K;
  const int tid = threadIdx.x;
  const int start = meta[L.seg_start + seg];
  const int len = meta[L.seg_len + seg];
  const int pos0 = meta[L.seg_pos0 + seg];
  const int pl = meta[L.req_prefix_len + j];
  const int ck = BRANCH ? -1 : meta[L.req_ckpt_pos + j];

  // history rows (raw inputs before the segment): trunk -> resume window or zeros;
  // question -> its request's trunk window (by index)
  const uint16_t* hist = nullptr;
  if (BRANCH) hist = p.hist_in;
  else if (pl > 0) hist = p.hist_in;
  const float* S0 = nullptr;
  if (BRANCH) S0 = p.state_in;
  else if (pl > 0) S0 = p.state_in;
  if (!BRANCH && pl > 0 && (!p.state_in || !p.hist_in)) {
    if (tid == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_BAD_PREFIX);
    return;
  }

  auto raw = [&](int o_seg, int s, int c) -> float {
    // raw input of stream s (0 q, 1 k, 2 v), channel c, at segment offset o_seg (may be < 0)
    if (o_seg >= 0) {
      const uint16_t* x = s == 0 ? p.q : (s == 1 ? p.k : p.v);
      return bf2f(x[(static_cast<int64_t>(start + o_seg) * H + h) * D + c]);
    }
    const int r = K - 1 + o_seg;
    if (r < 0 || hist == nullptr) return 0.f;
    return bf2f(hist[((static_cast<int64_t>(j * (K - 1) + r) * 3 + s) * H + h) * D + c]);
  };
  auto conv = [&](int o_seg, int s, int c) -> float {
    const float* w = p.conv_w + ((static_cast<int64_t>(s) * H + h) * D + c) * K;
    float y = 0.f;
    for (int i = 0; i < K; ++i) y += w[i] * raw(o_seg - (K - 1) + i, s, c);
    return y / (1.f + expf(-y));  // SiLU
  };

  // initial state slice
  for (int e = tid; e < DVS * D; e += NT) {
    const int r = e / D, c = e % D;
    sm.S[r * LDD + c] =
        S0 ? S0[((static_cast<int64_t>(j) * H + h) * D + z * DVS + r) * D + c] : 0.f;
  }
  __syncthreads();
  if (!BRANCH && ck >= 0 && ck - pos0 == 0 && p.S_ckpt) {
    for (int e = tid; e < DVS * D; e += NT) {
      const int r = e / D, c = e % D;
      p.S_ckpt[((static_cast<int64_t>(j) * H + h) * D + z * DVS + r) * D + c] = sm.S[r * LDD + c];
    }
  }

  for (int c0 = 0; c0 < len; c0 += C) {
    const int n = min(C, len - c0);
    // ---- gates ---------------------------------------------------------------
    if (tid < C) {
      const int u = tid;
      const int64_t row = static_cast<int64_t>(start + c0 + u) * H + h;
      sm.ETA[u] = u < n ? p.eta[row] : 0.f;
      sm.G[u] = u < n ? logf(p.alpha[row]) : 0.f;
    }
    __syncthreads();
    if (tid == 0) {
      float acc = 0.f;
      for (int u = 0; u < C; ++u) {
        acc += sm.G[u];
        sm.G[u] = acc;
        sm.EG[u] = expf(acc);
      }
      for (int u = 0; u < C; ++u) sm.GL[u] = expf(acc - sm.G[u]);
    }
    // ---- conv + SiLU ----------------------------------------------------------
    for (int e = tid; e < C * D; e += NT) {
      const int u = e / D, c = e % D;
      const bool ok = u < n;
      sm.Q[u * LDD + c] = ok ? conv(c0 + u, 0, c) : 0.f;
      sm.K[u * LDD + c] = ok ? conv(c0 + u, 1, c) : 0.f;
    }
    for (int e = tid; e < C * DVS; e += NT) {
      const int u = e / DVS, c = e % DVS;
      sm.U[u * LDV + c] = u < n ? conv(c0 + u, 2, z * DVS + c) : 0.f;
    }
    __syncthreads();
    // ---- L2 normalisation of q and k rows (one warp per row) -------------------
    {
      const int warp = tid >> 5, lane = tid & 31;
      for (int u = warp; u < 2 * C; u += NT / 32) {
        float* row = (u < C) ? &sm.Q[u * LDD] : &sm.K[(u - C) * LDD];
        float ss = 0.f;
        for (int c = lane; c < D; c += 32) ss += row[c] * row[c];
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = 1.f / sqrtf(ss + 1e-6f);
        for (int c = lane; c < D; c += 32) row[c] *= inv;
      }
    }
    __syncthreads();
    // RHS: W <- eta e^G K, U <- eta V
    for (int e = tid; e < C * D; e += NT) {
      const int u = e / D, c = e % D;
      sm.W[u * LDD + c] = sm.ETA[u] * sm.EG[u] * sm.K[u * LDD + c];
    }
    for (int e = tid; e < C * DVS; e += NT) {
      const int u = e / DVS, c = e % DVS;
      sm.U[u * LDV + c] *= sm.ETA[u];
    }
    // ---- Gram and query-key matrices -------------------------------------------
    for (int e = tid; e < C * C; e += NT) {
      const int t = e / C, s = e % C;
      float kk = 0.f, qk = 0.f;
      if (s <= t) {
        for (int c = 0; c < D; ++c) {
          const float ks = sm.K[s * LDD + c];
          kk += sm.K[t * LDD + c] * ks;
          qk += sm.Q[t * LDD + c] * ks;
        }
      }
      const float gam = s <= t ? expf(sm.G[t] - sm.G[s]) : 0.f;
      sm.A[t * LDC + s] = s < t ? sm.ETA[t] * gam * kk : 0.f;
      sm.QK[t * LDC + s] = gam * qk;
    }
    __syncthreads();
    // ---- forward substitution (I + A) X = RHS, one column per thread ------------
    if (tid < D + DVS) {
      float* X;
      int ld, c;
      if (tid < D) { X = sm.W; ld = LDD; c = tid; }
      else { X = sm.U; ld = LDV; c = tid - D; }
      for (int t = 1; t < C; ++t) {
        float acc = X[t * ld + c];
        for (int s = 0; s < t; ++s) acc -= sm.A[t * LDC + s] * X[s * ld + c];
        X[t * ld + c] = acc;
      }
    }
    __syncthreads();
    // ---- U = U~ - W S0^T ----------------------------------------------------------
    for (int e = tid; e < C * DVS; e += NT) {
      const int t = e / DVS, r = e % DVS;
      float acc = 0.f;
      for (int c = 0; c < D; ++c) acc += sm.W[t * LDD + c] * sm.S[r * LDD + c];
      sm.U[t * LDV + r] -= acc;
    }
    __syncthreads();
    // ---- outputs: O = e^G Q S0^T + (tril(Gamma) * QK^T) U ---------------------------
    for (int e = tid; e < C * DVS; e += NT) {
      const int t = e / DVS, r = e % DVS;
      if (t >= n) continue;
      float acc = 0.f;
      for (int c = 0; c < D; ++c) acc += sm.Q[t * LDD + c] * sm.S[r * LDD + c];
      acc *= sm.EG[t];
      for (int s = 0; s <= t; ++s) acc += sm.QK[t * LDC + s] * sm.U[s * LDV + r];
      p.o[(static_cast<int64_t>(start + c0 + t) * H + h) * D + z * DVS + r] = f2bf(acc);
    }
    // ---- checkpoint inside this chunk: state after r_ck tokens of it --------------
    if (!BRANCH && ck >= 0 && p.S_ckpt) {
      const int r_ck = ck - pos0 - c0;
      if (r_ck >= 1 && r_ck <= n) {
        const float gl = sm.G[r_ck - 1];
        for (int e = tid; e < DVS * D; e += NT) {
          const int r = e / D, c = e % D;
          float acc = expf(gl) * sm.S[r * LDD + c];
          for (int s = 0; s < r_ck; ++s)
            acc += expf(gl - sm.G[s]) * sm.U[s * LDV + r] * sm.K[s * LDD + c];
          p.S_ckpt[((static_cast<int64_t>(j) * H + h) * D + z * DVS + r) * D + c] = acc;
        }
      }
    }
    __syncthreads();
    // ---- state update: S = e^{G_last} S + U^T diag(Gamma_last,.) K ------------------
    {
      const float egl = sm.EG[C - 1];
      for (int e = tid; e < DVS * D; e += NT) {
        const int r = e / D, c = e % D;
        float acc = egl * sm.S[r * LDD + c];
        for (int s = 0; s < n; ++s) acc += sm.GL[s] * sm.U[s * LDV + r] * sm.K[s * LDD + c];
        sm.S[r * LDD + c] = acc;
      }
    }
    __syncthreads();
  }

  if (!BRANCH) {
    for (int e = tid; e < DVS * D; e += NT) {
      const int r = e / D, c = e % D;
      p.S_P[((static_cast<int64_t>(j) * H + h) * D + z * DVS + r) * D + c] = sm.S[r * LDD + c];
    }
    if (z == 0) {
      // conv windows: raw inputs of the last K-1 positions before the end / before m
      for (int e = tid; e < (K - 1) * 3 * D; e += NT) {
        const int i = e / (3 * D), s = (e / D) % 3, c = e % D;
        const int64_t dst = ((static_cast<int64_t>(j * (K - 1) + i) * 3 + s) * H + h) * D + c;
        p.conv_win[dst] = f2bf(raw(len - (K - 1) + i, s, c));
        if (ck >= 0 && p.conv_ckpt) p.conv_ckpt[dst] = f2bf(raw(ck - pos0 - (K - 1) + i, s, c));
      }
    }
  }
}

template <int D, bool BRANCH>
static int launch_gdn(const GdnParams& p, int grid_x, cudaStream_t s) {
  const size_t smem = sizeof(GdnSmem<D>);
  if (cudaFuncSetAttribute(gdn_chunk_kernel<D, BRANCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return FORK_ECUDA;
  dim3 grid(grid_x, p.H, D / DVS);
  gdn_chunk_kernel<D, BRANCH><<<grid, NT, smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? FORK_OK : FORK_ECUDA;
}

static int gdn_common_checks(const fork_meta* m, MetaLayout* L, const uint16_t* q, const uint16_t* k,
                             const uint16_t* v, const float* alpha, const float* eta,
                             const float* conv_w, int32_t H, int32_t d, int32_t K, int32_t chunk,
                             const uint16_t* o) {
  int rc = check_meta(m, L);
  if (rc != FORK_OK) return rc;
  if (!q || !k || !v || !alpha || !eta || !conv_w || !o) return FORK_EINVAL;
  if (H < 1 || (d != 64 && d != 128) || K != 4 || chunk != C) return FORK_EINVAL;
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
  (void)flags;
  MetaLayout L;
  int rc = gdn_common_checks(m, &L, q, k, v, alpha, eta, conv_w, H, d, K, chunk, o);
  if (rc != FORK_OK) return rc;
  if (!S_P || !conv_win) return FORK_EINVAL;
  if ((S_ckpt == nullptr) != (conv_ckpt == nullptr)) return FORK_EINVAL;
  if ((init_state == nullptr) != (init_conv == nullptr)) return FORK_EINVAL;
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
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return d == 64 ? launch_gdn<64, false>(p, m->max_req, s) : launch_gdn<128, false>(p, m->max_req, s);
}

extern "C" int fork_gdn_branches(const fork_meta* m, const uint16_t* q, const uint16_t* k,
                                 const uint16_t* v, const float* alpha, const float* eta,
                                 const float* conv_w, int32_t H, int32_t d, int32_t K,
                                 int32_t chunk, const float* S_P, const uint16_t* conv_win,
                                 uint16_t* o, uint32_t flags, void* stream) {
  (void)flags;
  MetaLayout L;
  int rc = gdn_common_checks(m, &L, q, k, v, alpha, eta, conv_w, H, d, K, chunk, o);
  if (rc != FORK_OK) return rc;
  if (!S_P || !conv_win) return FORK_EINVAL;
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
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return d == 64 ? launch_gdn<64, true>(p, m->max_q, s) : launch_gdn<128, true>(p, m->max_q, s);
}
