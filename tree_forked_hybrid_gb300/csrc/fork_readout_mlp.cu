// Selective readout with the final pointwise block on the question rows only
// (onedev summary "어떻게 쓰나": in the last layer the MLP and what follows run
// only on each question's last-token row, which changes no output).  With h_i
// the hidden row of question i's last stream token (metadata q_last):
//   n_i = bf16(rmsnorm(h_i) * g1)
//   a_i = bf16(silu(W_gate n_i) * (W_up n_i))          (SwiGLU, F wide)
//   y_i = h_i + W_down a_i
//   z_i = rmsnorm(y_i) * g2,   p_i(o) = softmax_{o in O_i}(w_o . z_i)   (eq. (1))
// rmsnorm(x) = x * (mean x^2 + 1e-6)^(-1/2).  Kernels: ro_norm_kernel (gather and
// norm, a CTA per question), ro_gemm_kernel (bf16 warp-MMA products over the
// question rows, each weight tile read once per 64-row tile: gate and up with the
// SwiGLU epilogue, then down with the residual), ro_final_kernel (final norm and
// eq. (1)).  Reductions run in a fixed order: a question's result does not depend
// on the rest of the round.
#include "fork_common.cuh"

namespace fork {

namespace {

constexpr int kMT = 64;    // question rows per tile (4 warps x 16)
constexpr int kNT = 32;    // output columns per CTA
constexpr int kKC = 64;    // k per stage
constexpr int kLD = kKC + 8;  // padded smem row (bf16): fragment loads hit 32 different banks
constexpr float kEps = 1e-6f;

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// sum over the block (256 threads), fixed order
__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int s = 16; s > 0; s >>= 1) v += __shfl_xor_sync(0xffffffffu, v, s);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += red[i];
  return t;
}

}  // namespace

// Rows of the block: the questions' last rows (selective readout), or every stream row.
__device__ __forceinline__ int ro_rows(const int32_t* meta, int all) { return all ? meta[H_T] : meta[H_NQ]; }
__device__ __forceinline__ int ro_src(const int32_t* meta, const MetaLayout& L, int all, int i) {
  return all ? i : meta[L.q_last + i];
}

// n_i = bf16(rmsnorm(h_{row(i)}) * g1) into row i of A [Mpad, D]
__global__ void __launch_bounds__(256) ro_norm_kernel(const int32_t* __restrict__ meta, MetaLayout L,
                                                      const uint16_t* __restrict__ h, int D,
                                                      const float* __restrict__ g1, uint16_t* __restrict__ A,
                                                      int all) {
  __shared__ float red[8];
  if (meta[H_VALID] == 0) return;
  const int i = blockIdx.x;
  if (i >= ro_rows(meta, all)) return;
  const uint16_t* x = h + static_cast<int64_t>(ro_src(meta, L, all, i)) * D;
  float ss = 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    const float v = bf2f(x[d]);
    ss += v * v;
  }
  const float inv = 1.f / sqrtf(block_sum(ss, red) / static_cast<float>(D) + kEps);
  for (int d = threadIdx.x; d < D; d += blockDim.x) A[static_cast<int64_t>(i) * D + d] = f2bf(bf2f(x[d]) * inv * g1[d]);
}

// C[r, n] over the question rows r of one 64-row tile and 32 columns n:
//   GLU:  out_bf16[r, n] = bf16(silu(A W0^T) * (A W1^T))
//   else: out_f32[r, n]  = A W0^T + h_{q_last(r)}[n]
// A [Mpad, K] bf16, W0/W1 [N, K] bf16 (K contiguous).  Rows r >= Nq read zeros and
// are not stored.  4 warps, warp w owns rows 16w..16w+15; m16n8k16 bf16 MMAs.
template <bool GLU>
__global__ void __launch_bounds__(128) ro_gemm_kernel(const int32_t* __restrict__ meta, MetaLayout L,
                                                      const uint16_t* __restrict__ A, int K, int N,
                                                      const uint16_t* __restrict__ W0,
                                                      const uint16_t* __restrict__ W1,
                                                      uint16_t* __restrict__ out_bf16, float* __restrict__ out_f32,
                                                      const uint16_t* __restrict__ h, int all) {
  constexpr int NW = GLU ? 2 : 1;
  __shared__ __align__(16) uint16_t As[2][kMT][kLD];
  __shared__ __align__(16) uint16_t Ws[2][NW][kNT][kLD];
  if (meta[H_VALID] == 0) return;
  const int nq = ro_rows(meta, all);
  const int m0 = blockIdx.y * kMT, n0 = blockIdx.x * kNT;
  if (m0 >= nq) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;

  auto load = [&](int stage, int k0) {
    // A: 64 rows x 8 pieces of 16 bytes; W: NW x 32 rows x 8 pieces
    for (int e = tid; e < kMT * 8; e += 128) {
      const int r = e >> 3, pc = e & 7;
      const bool ok = m0 + r < nq;
      const uint16_t* src = A + static_cast<int64_t>(ok ? m0 + r : 0) * K + k0 + pc * 8;
      cp_async16(&As[stage][r][pc * 8], src, ok);
    }
    for (int e = tid; e < NW * kNT * 8; e += 128) {
      const int mtx = e / (kNT * 8), r = (e >> 3) % kNT, pc = e & 7;
      const uint16_t* W = mtx == 0 ? W0 : W1;
      cp_async16(&Ws[stage][mtx][r][pc * 8], W + static_cast<int64_t>(n0 + r) * K + k0 + pc * 8, true);
    }
    asm volatile("cp.async.commit_group;\n" ::);
  };

  float acc[NW][4][4];
#pragma unroll
  for (int m = 0; m < NW; ++m)
#pragma unroll
    for (int nb = 0; nb < 4; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[m][nb][e] = 0.f;

  const int nk = K / kKC;
  load(0, 0);
  for (int kc = 0; kc < nk; ++kc) {
    const int st = kc & 1;
    if (kc + 1 < nk) {
      load(st ^ 1, (kc + 1) * kKC);
      asm volatile("cp.async.wait_group 1;\n" ::);
    } else {
      asm volatile("cp.async.wait_group 0;\n" ::);
    }
    __syncthreads();
    const int r0 = warp * 16;
#pragma unroll
    for (int ks = 0; ks < kKC / 16; ++ks) {
      const int kk = ks * 16 + 2 * t;
      uint32_t a[4];
      a[0] = *reinterpret_cast<const uint32_t*>(&As[st][r0 + g][kk]);
      a[1] = *reinterpret_cast<const uint32_t*>(&As[st][r0 + g + 8][kk]);
      a[2] = *reinterpret_cast<const uint32_t*>(&As[st][r0 + g][kk + 8]);
      a[3] = *reinterpret_cast<const uint32_t*>(&As[st][r0 + g + 8][kk + 8]);
#pragma unroll
      for (int m = 0; m < NW; ++m)
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&Ws[st][m][nb * 8 + g][kk]);
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&Ws[st][m][nb * 8 + g][kk + 8]);
          mma16816(acc[m][nb], a, b0, b1);
        }
    }
    __syncthreads();  // the stage is reloaded next iteration
  }

  // epilogue: c0, c1 at (row g, cols 2t, 2t+1), c2, c3 at (row g+8, same cols)
#pragma unroll
  for (int nb = 0; nb < 4; ++nb) {
    const int col = n0 + nb * 8 + 2 * t;
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      const int row = m0 + warp * 16 + g + 8 * hlf;
      if (row >= nq) continue;
      const float c0 = acc[0][nb][2 * hlf], c1 = acc[0][nb][2 * hlf + 1];
      if (GLU) {
        const float u0 = acc[NW - 1][nb][2 * hlf], u1 = acc[NW - 1][nb][2 * hlf + 1];
        const float s0 = c0 / (1.f + __expf(-c0)), s1 = c1 / (1.f + __expf(-c1));
        *reinterpret_cast<uint32_t*>(out_bf16 + static_cast<int64_t>(row) * N + col) = pack2(s0 * u0, s1 * u1);
      } else {
        const uint32_t hv =
            *reinterpret_cast<const uint32_t*>(h + static_cast<int64_t>(ro_src(meta, L, all, row)) * N + col);
        float2 y;
        y.x = c0 + bf2f(static_cast<uint16_t>(hv & 0xffffu));
        y.y = c1 + bf2f(static_cast<uint16_t>(hv >> 16));
        *reinterpret_cast<float2*>(out_f32 + static_cast<int64_t>(row) * N + col) = y;
      }
    }
  }
}

// z_i = rmsnorm(y_i) * g2 (shared memory), then eq. (1) over the question's options
__global__ void __launch_bounds__(256) ro_final_kernel(const int32_t* __restrict__ meta, const float* __restrict__ Y,
                                                       int D, const float* __restrict__ g2,
                                                       const uint16_t* __restrict__ w,
                                                       const int32_t* __restrict__ off, float* __restrict__ p) {
  extern __shared__ float z[];
  __shared__ float red[8];
  if (meta[H_VALID] == 0) return;
  const int i = blockIdx.x;
  if (i >= meta[H_NQ]) return;
  const float* y = Y + static_cast<int64_t>(i) * D;
  float ss = 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x) ss += y[d] * y[d];
  const float inv = 1.f / sqrtf(block_sum(ss, red) / static_cast<float>(D) + kEps);
  for (int d = threadIdx.x; d < D; d += blockDim.x) z[d] = y[d] * inv * g2[d];
  __syncthreads();
  const int a = off[i], b = off[i + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = a + warp; o < b; o += blockDim.x / 32) {
    const uint16_t* wr = w + static_cast<int64_t>(o) * D;
    float acc = 0.f;
    for (int d = 2 * lane; d < D; d += 64) {
      const uint32_t wv = *reinterpret_cast<const uint32_t*>(wr + d);
      acc += bf2f(static_cast<uint16_t>(wv & 0xffffu)) * z[d] + bf2f(static_cast<uint16_t>(wv >> 16)) * z[d + 1];
    }
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) p[o] = acc;
  }
  __syncthreads();
  if (warp == 0) {
    float mx = -INFINITY;
    for (int o = a + lane; o < b; o += 32) mx = fmaxf(mx, p[o]);
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    float sum = 0.f;
    for (int o = a + lane; o < b; o += 32) sum += expf(p[o] - mx);
    for (int s = 16; s > 0; s >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, s);
    const float inv_s = 1.f / sum;
    __syncwarp();
    for (int o = a + lane; o < b; o += 32) p[o] = expf(p[o] - mx) * inv_s;
  }
}

// z_r = bf16(rmsnorm(y_r) * g2) for every stream row r (the block on all rows)
__global__ void __launch_bounds__(256) ro_znorm_kernel(const int32_t* __restrict__ meta, const float* __restrict__ Y,
                                                       int D, const float* __restrict__ g2, uint16_t* __restrict__ z) {
  __shared__ float red[8];
  if (meta[H_VALID] == 0) return;
  const int r = blockIdx.x;
  if (r >= meta[H_T]) return;
  const float* y = Y + static_cast<int64_t>(r) * D;
  float ss = 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x) ss += y[d] * y[d];
  const float inv = 1.f / sqrtf(block_sum(ss, red) / static_cast<float>(D) + kEps);
  for (int d = threadIdx.x; d < D; d += blockDim.x) z[static_cast<int64_t>(r) * D + d] = f2bf(y[d] * inv * g2[d]);
}

struct RoWs {
  size_t a1, a2, y, total;
};
static RoWs ro_ws(int64_t max_q, int64_t D, int64_t F) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const int64_t M = (max_q + kMT - 1) / kMT * kMT;
  RoWs r;
  r.a1 = 0;
  r.a2 = al(r.a1 + static_cast<size_t>(M * D * 2));
  r.y = al(r.a2 + static_cast<size_t>(M * F * 2));
  r.total = al(r.y + static_cast<size_t>(M * D * 4));
  return r;
}

}  // namespace fork

using namespace fork;

extern "C" size_t fork_readout_mlp_workspace_bytes(int32_t max_q, int32_t D, int32_t F) {
  if (max_q < 0 || D < 64 || D % 64 != 0 || D > 8192 || F < 64 || F % 64 != 0 || F > 65536) return 0;
  return ro_ws(max_q, D, F).total;
}

extern "C" int fork_readout_mlp(const fork_meta* m, const uint16_t* h, int32_t D, int32_t F, const float* g1,
                                const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                                const float* g2, const uint16_t* w_opt, const int32_t* opt_off, float* p,
                                void* workspace, size_t ws_bytes, uint32_t flags, void* stream) {
  (void)flags;
  MetaLayout L;
  int rc = check_meta(m, &L);
  if (rc != FORK_OK) return rc;
  if (!h || !g1 || !w_gate || !w_up || !w_down || !g2 || !w_opt || !opt_off || !p || !workspace) return FORK_EINVAL;
  if (D < 64 || D % 64 != 0 || D > 8192 || F < 64 || F % 64 != 0 || F > 65536) return FORK_EINVAL;
  if (!is_aligned16(h) || !is_aligned16(w_gate) || !is_aligned16(w_up) || !is_aligned16(w_down) ||
      !is_aligned16(w_opt) || !is_aligned16(workspace))
    return FORK_EINVAL;
  const RoWs w = ro_ws(m->max_q, D, F);
  if (ws_bytes < w.total) return FORK_EINVAL;
  if ((rc = check_device()) != FORK_OK) return rc;
  if (m->max_q == 0) return FORK_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  uint16_t* a1 = reinterpret_cast<uint16_t*>(ws + w.a1);
  uint16_t* a2 = reinterpret_cast<uint16_t*>(ws + w.a2);
  float* y = reinterpret_cast<float*>(ws + w.y);
  const int32_t* meta = static_cast<const int32_t*>(m->d_buf);
  const int mt = (m->max_q + kMT - 1) / kMT;
  ro_norm_kernel<<<m->max_q, 256, 0, s>>>(meta, L, h, D, g1, a1, 0);
  ro_gemm_kernel<true><<<dim3(F / kNT, mt), 128, 0, s>>>(meta, L, a1, D, F, w_gate, w_up, a2, nullptr, nullptr, 0);
  ro_gemm_kernel<false><<<dim3(D / kNT, mt), 128, 0, s>>>(meta, L, a2, F, D, w_down, nullptr, nullptr, y, h, 0);
  const int zbytes = D * 4;
  if (zbytes > 48 * 1024 &&
      cuda_rc(cudaFuncSetAttribute(ro_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, zbytes)) != FORK_OK)
    return FORK_ECUDA;
  ro_final_kernel<<<m->max_q, 256, zbytes, s>>>(meta, y, D, g2, w_opt, opt_off, p);
  return cuda_rc(cudaGetLastError());
}

extern "C" size_t fork_pointwise_rows_workspace_bytes(int32_t T_cap, int32_t D, int32_t F) {
  if (T_cap < 1 || D < 64 || D % 64 != 0 || D > 8192 || F < 64 || F % 64 != 0 || F > 65536) return 0;
  return ro_ws(T_cap, D, F).total;
}

extern "C" int fork_pointwise_rows(const fork_meta* m, const uint16_t* h, int32_t D, int32_t F, const float* g1,
                                   const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                                   const float* g2, uint16_t* z, void* workspace, size_t ws_bytes, uint32_t flags,
                                   void* stream) {
  (void)flags;
  MetaLayout L;
  int rc = check_meta(m, &L);
  if (rc != FORK_OK) return rc;
  if (!h || !g1 || !w_gate || !w_up || !w_down || !g2 || !z || !workspace) return FORK_EINVAL;
  if (D < 64 || D % 64 != 0 || D > 8192 || F < 64 || F % 64 != 0 || F > 65536) return FORK_EINVAL;
  if (!is_aligned16(h) || !is_aligned16(w_gate) || !is_aligned16(w_up) || !is_aligned16(w_down) ||
      !is_aligned16(z) || !is_aligned16(workspace))
    return FORK_EINVAL;
  const RoWs w = ro_ws(L.T_cap, D, F);
  if (ws_bytes < w.total) return FORK_EINVAL;
  if ((rc = check_device()) != FORK_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  uint16_t* a1 = reinterpret_cast<uint16_t*>(ws + w.a1);
  uint16_t* a2 = reinterpret_cast<uint16_t*>(ws + w.a2);
  float* y = reinterpret_cast<float*>(ws + w.y);
  const int32_t* meta = static_cast<const int32_t*>(m->d_buf);
  const int mt = (L.T_cap + kMT - 1) / kMT;
  ro_norm_kernel<<<L.T_cap, 256, 0, s>>>(meta, L, h, D, g1, a1, 1);
  ro_gemm_kernel<true><<<dim3(F / kNT, mt), 128, 0, s>>>(meta, L, a1, D, F, w_gate, w_up, a2, nullptr, nullptr, 1);
  ro_gemm_kernel<false><<<dim3(D / kNT, mt), 128, 0, s>>>(meta, L, a2, F, D, w_down, nullptr, nullptr, y, h, 1);
  ro_znorm_kernel<<<L.T_cap, 256, 0, s>>>(meta, y, D, g2, z);
  return cuda_rc(cudaGetLastError());
}
