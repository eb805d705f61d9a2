// Selective readout with the final pointwise block on the question rows only
// (onedev summary "어떻게 쓰나": in the last layer the MLP and what follows run
// only on each question's last-token row, which changes no output).  With h_i
// the hidden row of question i's last stream token (metadata q_last):
//   n_i = bf16(rmsnorm(h_i) * g1)
//   a_i = bf16(silu(W_gate n_i) * (W_up n_i))          (SwiGLU, F wide)
//   y_i = h_i + W_down a_i
//   z_i = rmsnorm(y_i) * g2,   p_i(o) = softmax_{o in O_i}(w_o . z_i)   (eq. (1))
// rmsnorm(x) = x * (mean x^2 + 1e-6)^(-1/2).  Kernels: ro_norm_kernel (gather and
// norm, a CTA per question); ro_tc_kernel (tcgen05 products with the weight tile as
// the A operand, 128 output columns per CTA, and the question rows as the B operand,
// 64 per tile: each weight byte is read once and the rows once per 128 columns; the
// down product's reduction is split over 4 CTAs) with ro_glu_kernel (SwiGLU);
// ro_final_kernel (the 4 partial products summed in order + the residual, final norm
// and eq. (1)).  ro_gemm_kernel (bf16 warp-MMA products, each weight tile
// read once per 64-row tile) serves the block on every stream row and shapes the
// tcgen05 tiles do not divide.  Reductions run in a fixed order: a question's result
// does not depend on the rest of the round.
#include <algorithm>

#include "fork_attn.cuh"
#include "tc_ptx.cuh"

namespace fork {

namespace {

constexpr int kMT = 64;    // question rows per tile (4 warps x 16)
constexpr int kNT = 32;    // output columns per CTA
constexpr int kKC = 64;    // k per stage
constexpr int kLD = kKC + 8;  // padded smem row (bf16): fragment loads hit 32 different banks
constexpr float kEps = 1e-6f;
// tcgen05 products of the selective block
constexpr int kTcCols = 128;                  // output columns per CTA (MMA M)
constexpr int kTcRows = 64;                   // question rows per tile (MMA N)
constexpr int kTcK = 64;                      // k per stage: one 128-byte swizzled box
constexpr int kTcStages = 6;
constexpr int kTcWBox = kTcCols * 128;        // 16 KB
constexpr int kTcStage = kTcWBox + kTcRows * 128;  // + 8 KB of question rows
constexpr int kTcSplit = 4;                   // down product: reduction split over 4 CTAs
constexpr int kTcSmem = kTcStages * kTcStage + 256 + 1024;

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
  // 8 elements (16 bytes) per access; every access of a pass issued before its sums
  const uint4* x4 = reinterpret_cast<const uint4*>(h + static_cast<int64_t>(ro_src(meta, L, all, i)) * D);
  const int nc = D / 8;
  float ss = 0.f;
  for (int c = threadIdx.x; c < nc; c += blockDim.x) {
    const uint4 v = x4[c];
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float lo = __uint_as_float(wv[q] << 16), hi = __uint_as_float(wv[q] & 0xffff0000u);
      ss = fmaf(lo, lo, fmaf(hi, hi, ss));
    }
  }
  const float inv = 1.f / sqrtf(block_sum(ss, red) / static_cast<float>(D) + kEps);
  const float4* g4 = reinterpret_cast<const float4*>(g1);
  uint4* a4 = reinterpret_cast<uint4*>(A + static_cast<int64_t>(i) * D);
  for (int c = threadIdx.x; c < nc; c += blockDim.x) {
    const uint4 v = x4[c];
    const float4 ga = g4[2 * c], gb = g4[2 * c + 1];
    const float gv[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = pack2(__uint_as_float(wv[q] << 16) * inv * gv[2 * q], __uint_as_float(wv[q] & 0xffff0000u) * inv * gv[2 * q + 1]);
    a4[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
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

// P[z][r][n] = sum over k in this CTA's range of A[r][k] W[n][k] for the question rows r of
// row tile blockIdx.y (64) and the columns n0..n0+127 of blockIdx.x: the weight tile is the
// A operand of tcgen05.mma (M = 128), the question rows the B operand (N = 64), fp32 in
// TMEM.  z = blockIdx.z selects the matrix (wmap0 for z < ks, else wmap1) and the k slice
// z % ks of length k_len.  One thread loads (TMA, kTcStages-deep ring), one issues the
// products; all 128 threads then read TMEM (thread = output column) and store row by row.
// Rows past the question count are computed from whatever the row buffer holds there and not
// stored (rows are independent).  Every wait is bounded.
__global__ void __launch_bounds__(128, 1)
    ro_tc_kernel(const __grid_constant__ CUtensorMap wmap0, const __grid_constant__ CUtensorMap wmap1,
                 const __grid_constant__ CUtensorMap amap, const int32_t* __restrict__ meta, int N, int k_len, int ks,
                 float* __restrict__ P, int rows_pad, uint64_t wait_ns) {
  extern __shared__ __align__(1024) unsigned char ro_tc_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(ro_tc_raw) + 1023) &
                                                       ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kTcStages * kTcStage);  // FULL[s], EMPTY[s], DONE
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * kTcStages + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 2);
  if (meta[H_VALID] == 0) return;
  const int nq = meta[H_NQ];
  const int m0 = blockIdx.y * kTcRows;
  if (m0 >= nq) return;
  const int n0 = blockIdx.x * kTcCols;
  const int z = blockIdx.z, k0 = (z % ks) * k_len;
  const int nst = k_len / kTcK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 2 * kTcStages + 1; ++i) tc::mbar_init(&bars[i], 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, 64);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0) {
    // producer: weight box (64 k x 128 columns) and row box (64 k x 64 rows) per stage
    const CUtensorMap* wm = z < ks ? &wmap0 : &wmap1;
    tc::prefetch_tmap(wm);
    tc::prefetch_tmap(&amap);
    int issued = 0;
    for (int i = 0; i < nst; ++i) {
      const int s = i % kTcStages;
      if (i >= kTcStages && !tc::mbar_wait(&bars[kTcStages + s], ((i / kTcStages) - 1) & 1, abort, wait_ns)) break;
      unsigned char* st = sm + s * kTcStage;
      tc::mbar_expect_tx(&bars[s], kTcStage);
      tc::tma_load_3d(st, wm, &bars[s], k0 + i * kTcK, 0, n0);
      tc::tma_load_3d(st + kTcWBox, &amap, &bars[s], k0 + i * kTcK, 0, m0);
      issued = i + 1;
    }
    // the last copies into each slot complete by themselves
    for (int i = max(0, issued - kTcStages); i < issued; ++i) tc::mbar_drain(&bars[i % kTcStages], (i / kTcStages) & 1);
  } else if (tid == 32) {
    // products: 4 k steps of 16 per stage, +32 bytes each in both operands
    constexpr uint32_t idesc = tc::idesc_bf16(kTcCols, kTcRows, 0, 0);
    for (int i = 0; i < nst; ++i) {
      const int s = i % kTcStages;
      if (!tc::mbar_wait(&bars[s], (i / kTcStages) & 1, abort, wait_ns)) break;
      tc::tc_fence_after();
      const uint64_t da = tc::sdesc_sw128(tc::smem_u32(sm + s * kTcStage), 16, 1024);
      const uint64_t db = tc::sdesc_sw128(tc::smem_u32(sm + s * kTcStage + kTcWBox), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < kTcK / 16; ++kk) tc::mma_bf16(tmem, da + kk * 2, db + kk * 2, idesc, (i | kk) ? 1u : 0u);
      tc::mma_commit(&bars[kTcStages + s]);
    }
    tc::mma_commit(&bars[2 * kTcStages]);  // every product issued (also after an abort)
  }
  __syncwarp();
  // the products are complete before TMEM is read or released; every thread then sees the
  // same abort flag
  tc::mbar_drain(&bars[2 * kTcStages], 0);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const bool aborted = *abort != 0;
  if (!aborted) {
    const int n = n0 + warp * 32 + lane;
    float* out = P + static_cast<int64_t>(z) * rows_pad * N + n;
    const uint32_t lb = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll
    for (int c = 0; c < kTcRows; c += 32) {
      uint32_t v[32];
      tc::tmem_ld32(tmem + lb + c, v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (m0 + c + e < nq) out[static_cast<int64_t>(m0 + c + e) * N] = __uint_as_float(v[e]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (aborted && tid == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_TIMEOUT);
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 64);
  }
}

// a2[r][n] = bf16(silu(gate) * up), gate = P[0][r][n], up = P[1][r][n], for question rows r
__global__ void __launch_bounds__(256) ro_glu_kernel(const int32_t* __restrict__ meta, const float* __restrict__ P,
                                                     int F, int rows_pad, uint16_t* __restrict__ a2) {
  if (meta[H_VALID] == 0) return;
  const int64_t total = static_cast<int64_t>(meta[H_NQ]) * F;
  const int64_t plane = static_cast<int64_t>(rows_pad) * F;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float g = P[e], u = P[plane + e];
    a2[e] = f2bf(g / (1.f + __expf(-g)) * u);
  }
}

// z_i = rmsnorm(y_i) * g2 (shared memory), then eq. (1) over the question's options.  With
// partial products P (the tcgen05 path), y_i is first formed here as the sum of the
// kTcSplit partials in order plus h_{q_last(i)}, and stored to Y.
__global__ void __launch_bounds__(256) ro_final_kernel(const int32_t* __restrict__ meta, MetaLayout L,
                                                       float* __restrict__ Y, const float* __restrict__ P,
                                                       int rows_pad, const uint16_t* __restrict__ h, int D,
                                                       const float* __restrict__ g2,
                                                       const uint16_t* __restrict__ w,
                                                       const int32_t* __restrict__ off, float* __restrict__ p) {
  extern __shared__ float z[];
  __shared__ float red[8];
  if (meta[H_VALID] == 0) return;
  const int i = blockIdx.x;
  if (i >= meta[H_NQ]) return;
  // 16-byte accesses throughout: y and g2 as float4, option weights as 8 bf16
  float4* y4 = reinterpret_cast<float4*>(Y + static_cast<int64_t>(i) * D);
  const float4* g4 = reinterpret_cast<const float4*>(g2);
  float4* z4 = reinterpret_cast<float4*>(z);
  if (P) {
    const int64_t plane = static_cast<int64_t>(rows_pad) * D;
    const float4* p4 = reinterpret_cast<const float4*>(P + static_cast<int64_t>(i) * D);
    const uint2* h4 = reinterpret_cast<const uint2*>(h + static_cast<int64_t>(meta[L.q_last + i]) * D);
    for (int c = threadIdx.x; c < D / 4; c += blockDim.x) {
      float4 acc = p4[c];
#pragma unroll
      for (int k = 1; k < kTcSplit; ++k) {
        const float4 q = p4[k * plane / 4 + c];
        acc.x += q.x;
        acc.y += q.y;
        acc.z += q.z;
        acc.w += q.w;
      }
      const uint2 hv = h4[c];
      acc.x += __uint_as_float(hv.x << 16);
      acc.y += __uint_as_float(hv.x & 0xffff0000u);
      acc.z += __uint_as_float(hv.y << 16);
      acc.w += __uint_as_float(hv.y & 0xffff0000u);
      y4[c] = acc;  // read back below by the same thread
    }
  }
  float ss = 0.f;
  for (int c = threadIdx.x; c < D / 4; c += blockDim.x) {
    const float4 v = y4[c];
    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
  }
  const float inv = 1.f / sqrtf(block_sum(ss, red) / static_cast<float>(D) + kEps);
  for (int c = threadIdx.x; c < D / 4; c += blockDim.x) {
    const float4 v = y4[c], g = g4[c];
    z4[c] = make_float4(v.x * inv * g.x, v.y * inv * g.y, v.z * inv * g.z, v.w * inv * g.w);
  }
  __syncthreads();
  const int a = off[i], b = off[i + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = a + warp; o < b; o += blockDim.x / 32) {
    const uint4* w4 = reinterpret_cast<const uint4*>(w + static_cast<int64_t>(o) * D);
    float acc = 0.f;
#pragma unroll 4
    for (int c = lane; c < D / 8; c += 32) {
      const uint4 wv = w4[c];
      const float4 za = z4[2 * c], zb = z4[2 * c + 1];
      acc = fmaf(__uint_as_float(wv.x << 16), za.x, acc);
      acc = fmaf(__uint_as_float(wv.x & 0xffff0000u), za.y, acc);
      acc = fmaf(__uint_as_float(wv.y << 16), za.z, acc);
      acc = fmaf(__uint_as_float(wv.y & 0xffff0000u), za.w, acc);
      acc = fmaf(__uint_as_float(wv.z << 16), zb.x, acc);
      acc = fmaf(__uint_as_float(wv.z & 0xffff0000u), zb.y, acc);
      acc = fmaf(__uint_as_float(wv.w << 16), zb.z, acc);
      acc = fmaf(__uint_as_float(wv.w & 0xffff0000u), zb.w, acc);
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
  size_t a1, a2, y, part, total;
};
// rows A of the first product (a1), of the second (a2), y; for the tcgen05 path of the
// selective block also the partial products (max(2F, 4D) values per row)
static RoWs ro_ws(int64_t max_q, int64_t D, int64_t F, bool tc) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const int64_t M = (max_q + kMT - 1) / kMT * kMT;
  RoWs r;
  r.a1 = 0;
  r.a2 = al(r.a1 + static_cast<size_t>(M * D * 2));
  r.y = al(r.a2 + static_cast<size_t>(M * F * 2));
  r.part = al(r.y + static_cast<size_t>(M * D * 4));
  r.total = al(r.part + (tc ? static_cast<size_t>(M) * std::max<int64_t>(2 * F, kTcSplit * D) * 4 : 0));
  return r;
}
// the tcgen05 path takes D and F that its tiles divide
static bool ro_tc_shapes(int64_t D, int64_t F) {
  return D % kTcCols == 0 && F % kTcCols == 0 && F % (kTcSplit * kTcK) == 0;
}

}  // namespace fork

using namespace fork;

extern "C" size_t fork_readout_mlp_workspace_bytes(int32_t max_q, int32_t D, int32_t F) {
  if (max_q < 0 || D < 64 || D % 64 != 0 || D > 8192 || F < 64 || F % 64 != 0 || F > 65536) return 0;
  return ro_ws(max_q, D, F, ro_tc_shapes(D, F)).total;
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
      !is_aligned16(w_opt) || !is_aligned16(g1) || !is_aligned16(g2) || !is_aligned16(workspace))
    return FORK_EINVAL;
  const bool tc = ro_tc_shapes(D, F);
  const RoWs w = ro_ws(m->max_q, D, F, tc);
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
  if (tc) {
    // tensor maps: weights [N rows, K] and question rows [mt * 64, K], 64-element boxes
    const int rows_pad = mt * kMT;
    float* part = reinterpret_cast<float*>(ws + w.part);
    alignas(64) CUtensorMap mg, mu, md, ma1, ma2;
    if (!encode_map_3d(&mg, w_gate, D, 1, F, kTcK, 1, kTcCols, true) ||
        !encode_map_3d(&mu, w_up, D, 1, F, kTcK, 1, kTcCols, true) ||
        !encode_map_3d(&md, w_down, F, 1, D, kTcK, 1, kTcCols, true) ||
        !encode_map_3d(&ma1, a1, D, 1, rows_pad, kTcK, 1, kTcRows, true) ||
        !encode_map_3d(&ma2, a2, F, 1, rows_pad, kTcK, 1, kTcRows, true))
      return FORK_ECUDA;
    static const int attr = [] {
      return cudaFuncSetAttribute(ro_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem) == cudaSuccess
                 ? static_cast<int>(FORK_OK)
                 : static_cast<int>(FORK_ECUDA);
    }();
    if (attr != FORK_OK) return attr;
    const uint64_t wns = wait_ns_of(m);
    const int eblocks = static_cast<int>(std::min<int64_t>((static_cast<int64_t>(m->max_q) * F + 255) / 256, 8 * sm_count()));
    ro_tc_kernel<<<dim3(F / kTcCols, mt, 2), 128, kTcSmem, s>>>(mg, mu, ma1, meta, F, D, 1, part, rows_pad, wns);
    ro_glu_kernel<<<std::max(eblocks, 1), 256, 0, s>>>(meta, part, F, rows_pad, a2);
    ro_tc_kernel<<<dim3(D / kTcCols, mt, kTcSplit), 128, kTcSmem, s>>>(md, md, ma2, meta, D, F / kTcSplit, kTcSplit,
                                                                       part, rows_pad, wns);
  } else {
    ro_gemm_kernel<true><<<dim3(F / kNT, mt), 128, 0, s>>>(meta, L, a1, D, F, w_gate, w_up, a2, nullptr, nullptr, 0);
    ro_gemm_kernel<false><<<dim3(D / kNT, mt), 128, 0, s>>>(meta, L, a2, F, D, w_down, nullptr, nullptr, y, h, 0);
  }
  const int zbytes = D * 4;
  if (zbytes > 48 * 1024 &&
      cuda_rc(cudaFuncSetAttribute(ro_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, zbytes)) != FORK_OK)
    return FORK_ECUDA;
  ro_final_kernel<<<m->max_q, 256, zbytes, s>>>(meta, L, y, tc ? reinterpret_cast<const float*>(ws + w.part) : nullptr,
                                                 mt * kMT, h, D, g2, w_opt, opt_off, p);
  return cuda_rc(cudaGetLastError());
}

extern "C" size_t fork_pointwise_rows_workspace_bytes(int32_t T_cap, int32_t D, int32_t F) {
  if (T_cap < 1 || D < 64 || D % 64 != 0 || D > 8192 || F < 64 || F % 64 != 0 || F > 65536) return 0;
  return ro_ws(T_cap, D, F, false).total;
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
      !is_aligned16(g1) || !is_aligned16(z) || !is_aligned16(workspace))
    return FORK_EINVAL;
  const RoWs w = ro_ws(L.T_cap, D, F, false);
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
