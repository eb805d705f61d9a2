// Two-call forked Gated DeltaNet on the 5th-generation tensor cores (tcgen05, TF32).
//
// Gated delta rule of the rainbus summary "前置知识", in the chunked form that the
// DFlash-TfM summary ("GDN을 위한 롤백 없는 트리 검증") solves with a Gram matrix and a
// triangular solve.  For a chunk of C = 64 tokens with start state S0 (d_v x d_k),
// G_t = sum_{s<=t} log a_s, Gamma_ts = exp(G_t - G_s),
//   A_ts = eta_t Gamma_ts k_t.k_s (s < t),  T = (I + A)^{-1}
//   W = T diag(eta e^G) K,  U~ = T diag(eta) V        (independent of S0)
//   U = U~ - W S0^T
//   O = diag(e^G) Q S0^T + (tril(Gamma) * Q K^T) U
//   S = e^{G_last} S0 + U^T diag(Gamma_last) K.
// Everything above the line "U = ..." depends only on the chunk's inputs, so it is
// prepared for chunk k+1 while the state of chunk k is being updated:
//
// One CTA = one trunk (call 1) or a group of up to kQG questions of one request
// (call 2) x one head; d = 128.  12 warps:
//   warps 0-7   prep: raw q/k/v rows by TMA (67 rows: the chunk and the three before
//               it), gates, causal conv + SiLU (eta V written straight into tensor
//               memory as an MMA operand), L2 norm, Q K^T products, P and A, T by
//               blocked forward substitution, then W^T = (eta e^G K)^T T^T and
//               U~^T = (eta V)^T T^T on the tensor cores; -W replaces K in the
//               operand tile.
//   warps 8-11  state chain (thread = TMEM lane = row v of S): U^T = U~^T - S W^T and
//               X = S Q^T (A operand S read from tensor memory), U^T rounded to TF32,
//               X scaled by e^G, S by e^{G_last}, then O^T = X + U^T P^T and
//               S += U^T diag(Gamma_last) K, and the output rows.
// S (128 x 128 fp32) stays in tensor memory for the whole segment.  Operands written
// by threads are rounded to TF32 (nearest); T is formed in fp32.  Every wait is
// bounded and agreed by the threads of its role.
#include "fork_attn.cuh"
#include "fork_gdn.cuh"
#include "tc_ptx.cuh"

namespace fork {

namespace {
constexpr int D = 128;
constexpr int C = 64;
constexpr int NT = 384;       // 8 prep warps + 4 chain warps
constexpr int NP = 256;       // prep threads
constexpr int NCH = 128;      // chain threads
constexpr int KW = 4;
constexpr int HR = C + KW - 1;  // raw rows staged per chunk
constexpr int LDC = C + 4;      // plain 64-wide fp32 tiles
constexpr int kQG = 4;          // questions per CTA in the branch call
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S, two (U, X) slots, eta V, Q K^T / (eta e^G K)^T
constexpr uint32_t T_S = 0, T_AV = 384, T_M1 = 448;
__device__ __forceinline__ uint32_t t_u(int slot) { return 128u + 128u * slot; }
__device__ __forceinline__ uint32_t t_x(int slot) { return 192u + 128u * slot; }

struct Lay {
  static constexpr int QK = 0;                 // [Q; K -> -W] 128 rows x 128 fp32 (4 boxes of 32 columns)
  static constexpr int KT = QK + 4 * 16384;    // diag(Gamma_last) K, transposed: 128 rows (d_k) x 64 (2 boxes)
  static constexpr int TB = KT + 2 * 16384;    // T: 64 x 64 (2 boxes)
  static constexpr int PB = TB + 2 * 8192;     // P: 64 x 64 (2 boxes)
  static constexpr int RAWS = HR * D * 2;      // one stream's raw rows (bf16)
  static constexpr int RAW = PB + 2 * 8192;    // [3][HR][D] bf16
  static constexpr int AM = RAW + 3 * RAWS;    // plain A [64][LDC]
  static constexpr int TM = AM + C * LDC * 4;  // plain T [64][LDC]
  static constexpr int XS = TM + C * LDC * 4;  // inverse scratch [3*256]
  static constexpr int GT = XS + 3 * 256 * 4;  // raw alpha, eta [2][64]; per slot G, EG, GL, ETA, IG [2][5][64]
  static constexpr int SEG = GT + (2 * C + 2 * 5 * C) * 4;  // this CTA's segments: start, len, pos0
  static constexpr int BAR = SEG + 64;
  static constexpr int BYTES = BAR + 256;
  static constexpr int SMEM = BYTES + 1024;
};
static_assert(Lay::SMEM <= 232448, "shared memory budget");
static_assert(3 * kQG * 4 <= 64, "segment table");
static_assert(Lay::RAW % 128 == 0 && Lay::RAWS % 128 == 0, "TMA destinations");

enum { B_RAW = 0, B_M1, B_MW, B_PREP, B_MA, B_MB, B_EPI0, B_EPI1, B_OUT, B_FINP, B_FINC, B_STALL, B_N };

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

// x rounded to TF32 (10-bit mantissa), to nearest with ties away from zero: add half
// a unit of the last kept place to the magnitude bits and clear the 13 dropped bits.
// Exact for finite x (a carry into the exponent is the correct rounding up); two
// integer operations instead of a conversion instruction.
__device__ __forceinline__ uint32_t tf32_bits(float x) {
  return (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
}
// byte offset of fp32 element (r, c) in a K-major 128-byte-swizzled tile of
// 32-column boxes of `rows` rows
__device__ __forceinline__ int swz(int rows, int r, int c) {
  const int cc = c & 31;
  return (c >> 5) * rows * 128 + r * 128 + ((((cc >> 2) ^ (r & 7))) << 4) + ((cc & 3) << 2);
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(tc::smem_u32(dst)), "l"(src),
               "r"(valid ? 4 : 0));
}
__device__ __forceinline__ float bf_at(const unsigned char* p) {
  return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
}
// 32 consecutive fp32 values (16-byte aligned) into registers with 8 vector loads
__device__ __forceinline__ void ld32f(const float* src, float* dst) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 v = reinterpret_cast<const float4*>(src)[q];
    dst[4 * q] = v.x;
    dst[4 * q + 1] = v.y;
    dst[4 * q + 2] = v.z;
    dst[4 * q + 3] = v.w;
  }
}
// barrier over the `n` threads of one role; returns true iff every one of them passed ok
__device__ __forceinline__ bool role_and(int id, int n, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(ok)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void role_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
}  // namespace

template <bool BRANCH>
__global__ void __launch_bounds__(NT, 1)
    gdn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const GdnParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int32_t* meta = p.meta;
  const MetaLayout& L = p.L;
  if (meta[H_VALID] == 0) return;
  const int R = meta[H_R];
  const int x = blockIdx.x;
  int seg_first, seg_end, j;
  if (BRANCH) {
    // the CTA of question x leads a group of up to kQG consecutive questions of its request
    if (x >= meta[H_NQ]) return;
    j = meta[L.seg_req + R + x];
    if (p.checks && (j < 0 || j >= R)) {
      if (threadIdx.x == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_CHECK);
      return;
    }
    const int fq = meta[L.req_first_q + j], nq = meta[L.req_n_q + j];
    if ((x - fq) % kQG != 0) return;
    seg_first = R + x;
    seg_end = R + min(x + kQG, fq + nq);
  } else {
    if (x >= R) return;
    j = x;
    seg_first = x;
    seg_end = x + 1;
  }
  if (p.checks && !gdn_segs_in_bounds(meta, L, seg_first, seg_end, j)) {
    if (threadIdx.x == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_CHECK);
    return;
  }
  const int h = blockIdx.y;
  const int H = p.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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

  unsigned char* qk = sm + Lay::QK;
  unsigned char* kt = sm + Lay::KT;
  unsigned char* tb = sm + Lay::TB;
  unsigned char* pb = sm + Lay::PB;
  unsigned char* raw = sm + Lay::RAW;
  float* am = reinterpret_cast<float*>(sm + Lay::AM);
  float* tm = reinterpret_cast<float*>(sm + Lay::TM);
  float* xs = reinterpret_cast<float*>(sm + Lay::XS);
  float* ga = reinterpret_cast<float*>(sm + Lay::GT);
  float* ge = ga + C;
  float* gslot = ge + C;  // [slot][G, EG, GL, ETA, IG][64]
  int* segt = reinterpret_cast<int*>(sm + Lay::SEG);  // [kQG][3], read instead of the metadata
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::BAR + B_N * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + Lay::BAR + B_N * 8 + 8);

  if (tid == 0) {
    // B_STALL is completed by nothing (FORK_TEST_STALL)
    for (int b = 0; b < B_N; ++b) tc::mbar_init(&bars[b], (b == B_EPI0 || b == B_EPI1 || b == B_OUT) ? NCH : 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (tid < seg_end - seg_first) {
    segt[3 * tid] = meta[L.seg_start + seg_first + tid];
    segt[3 * tid + 1] = meta[L.seg_len + seg_first + tid];
    segt[3 * tid + 2] = meta[L.seg_pos0 + seg_first + tid];
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  // a checkpoint at the first position of a trunk is its start state
  if (!BRANCH && ck >= 0 && p.S_ckpt && ck == meta[L.seg_pos0 + j]) {
    for (int e = tid; e < D * D; e += NT) p.S_ckpt[state_base + e] = S0 ? S0[state_base + e] : 0.f;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t qk_a = tc::smem_u32(qk), kt_a = tc::smem_u32(kt), tb_a = tc::smem_u32(tb),
                 pb_a = tc::smem_u32(pb);
  const int q4 = warp & 3;                                  // TMEM lane quarter of this warp
  const uint32_t lb = static_cast<uint32_t>(q4 * 32) << 16;  // its lane base
  auto seg_start = [&](int s) { return segt[3 * (s - seg_first)]; };
  auto seg_len = [&](int s) { return segt[3 * (s - seg_first) + 1]; };
  auto seg_pos0 = [&](int s) { return segt[3 * (s - seg_first) + 2]; };
  // first chunk at or after segment s
  auto first_seg = [&](int s) {
    while (s < seg_end && seg_len(s) == 0) ++s;
    return s;
  };

  if (warp < 8) {
    // ============================ prep (256 threads) ============================
    const int hf = warp >> 2;          // column / token half
    const int ch = q4 * 32 + lane;     // channel = TMEM lane of this thread
    const int u0 = hf * 32;            // first token of this thread's half
    auto pwait = [&](int b, uint32_t par) -> bool {
      return role_and(1, NP, tc::mbar_wait(&bars[b], par, abort, p.wait_ns));
    };
    // conv weights: the v stream for channel ch; q, k for the channel pair of the P4 mapping
    const int cp = (warp & 1) * 32 + lane, c2 = 2 * cp;
    float wv[KW], wq[2][2][KW];
#pragma unroll
    for (int i = 0; i < KW; ++i) wv[i] = p.conv_w[((static_cast<int64_t>(2) * H + h) * D + ch) * KW + i];
#pragma unroll
    for (int st = 0; st < 2; ++st)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int i = 0; i < KW; ++i)
          wq[st][cc][i] = p.conv_w[((static_cast<int64_t>(st) * H + h) * D + c2 + cc) * KW + i];
    // raw rows start-3 .. start+63 of the three streams (TMA; rows outside the tensor read
    // as zero) and the gates of a chunk
    const CUtensorMap* maps[3] = {&qmap, &kmap, &vmap};
    int raw_issued = 0;
    auto issue_loads = [&](int s, int cc) {
      const int st0 = seg_start(s), ln = seg_len(s);
      if (tid == 0) {
        tc::fence_proxy_async_smem();  // the rows were last read (and patched) by threads
        tc::mbar_expect_tx(&bars[B_RAW], 3 * Lay::RAWS);
#pragma unroll
        for (int st = 0; st < 3; ++st) tc::tma_load_3d(raw + st * Lay::RAWS, maps[st], &bars[B_RAW], 0, h, st0 + cc - (KW - 1));
      }
      ++raw_issued;
      if (tid < 2 * C) {
        const int u = tid & (C - 1);
        const bool valid = cc + u < ln;
        const float* src = (tid < C ? p.alpha : p.eta) + (static_cast<int64_t>(st0 + (valid ? cc + u : 0)) * H + h);
        cp_async4(tid < C ? &ga[u] : &ge[u], src, valid);
      }
      asm volatile("cp.async.commit_group;\n" ::);
    };
    if (tid == 0) {
      tc::prefetch_tmap(&qmap);
      tc::prefetch_tmap(&kmap);
      tc::prefetch_tmap(&vmap);
    }
    // blocks of T above the diagonal stay zero (the operand tile, and the blocks (0,1) and
    // (2,3) of the fp32 copy, which the two-level products read)
    for (int e = tid; e < C * C; e += NP) {
      const int t = e >> 6, s = e & 63;
      if ((s >> 4) > (t >> 4)) *reinterpret_cast<uint32_t*>(tb + swz(64, t, s)) = 0u;
      if ((s >> 4) == (t >> 4) + 1 && (t >> 4) % 2 == 0) tm[t * LDC + s] = 0.f;
    }
    bool ok = true;
    int si = first_seg(seg_first), c0 = 0, k = 0;
    if (si < seg_end) issue_loads(si, 0);
    while (ok && si < seg_end) {
      const int len = seg_len(si);
      const int n = min(C, len - c0);
      const int slot = k & 1;
      float* G = gslot + slot * 5 * C;
      float* EG = G + C;
      float* GL = EG + C;
      float* ETA = GL + C;
      float* IG = ETA + C;
      int nsi = si, nc0 = c0 + C;
      if (nc0 >= len) {
        nsi = first_seg(si + 1);
        nc0 = 0;
      }
      // ---- P0: this chunk's rows and gates have landed; history rows of a segment start
      if (!(ok = pwait(B_RAW, (raw_issued - 1) & 1))) break;
      asm volatile("cp.async.wait_group 0;\n" ::);
      if (c0 == 0) {
        for (int e = tid; e < 3 * (KW - 1) * D; e += NP) {
          const int st = e / ((KW - 1) * D), i = (e / D) % (KW - 1), c = e % D;
          const uint16_t hv =
              hist ? hist[((static_cast<int64_t>(j * (KW - 1) + i) * 3 + st) * H + h) * D + c] : uint16_t(0);
          *reinterpret_cast<uint16_t*>(raw + st * Lay::RAWS + i * D * 2 + c * 2) = hv;
        }
      }
      role_sync(1, NP);
      // ---- P1: gates (warp 0; SFU log and exp: the cumulative log gate is off by at most
      //      ~3e-5 over a chunk, far below the TF32 rounding of the operands it scales) ----
      if (warp == 0) {
        const int a0 = 2 * lane, a1 = a0 + 1;
        const float l0 = a0 < n ? __logf(ga[a0]) : 0.f, l1 = a1 < n ? __logf(ga[a1]) : 0.f;
        float xx = l0 + l1;
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, xx, o);
          if (lane >= o) xx += y;
        }
        const float g1 = xx, g0 = xx - l1;
        const float glast = __shfl_sync(0xffffffffu, xx, 31);
        G[a0] = g0;
        G[a1] = g1;
        EG[a0] = __expf(g0);
        EG[a1] = __expf(g1);
        GL[a0] = __expf(glast - g0);
        GL[a1] = __expf(glast - g1);
        ETA[a0] = a0 < n ? ge[a0] : 0.f;
        ETA[a1] = a1 < n ? ge[a1] : 0.f;
        IG[a0] = __expf(-g0);  // used only when no G of the chunk is below -80 (no overflow)
        IG[a1] = __expf(-g1);
      }
      role_sync(1, NP);
      // ---- P2: v stream: conv + SiLU, times eta, TF32, into TMEM (A operand of U~) ----
      {
        const unsigned char* col = raw + 2 * Lay::RAWS + ch * 2;
        float x0 = bf_at(col + (u0 + 0) * D * 2), x1 = bf_at(col + (u0 + 1) * D * 2), x2 = bf_at(col + (u0 + 2) * D * 2);
        uint32_t av[32];
        float etv[32];
        ld32f(ETA + u0, etv);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float x3 = bf_at(col + (u0 + e + 3) * D * 2);
          const float y = silu(wv[0] * x0 + wv[1] * x1 + wv[2] * x2 + wv[3] * x3);
          av[e] = (u0 + e < n) ? tf32_bits(etv[e] * y) : 0u;
          x0 = x1;
          x1 = x2;
          x2 = x3;
        }
        tc::tmem_st32(tmem + T_AV + u0 + lb, av);
      }
      // ---- P3: the operand tile is free once the chain's S [-W; Q]^T of chunk k-1 is done
      if (k >= 1 && !(ok = pwait(B_MA, (k - 1) & 1))) break;
      // ---- P4: q, k streams: conv + SiLU (fp32) into the [Q; K] tile; thread = channel
      //      pair (32 per warp: 128 contiguous bytes of a raw row) x 16 tokens --------------
      {
        const int ub = (warp >> 1) * 16;  // first token; channels c2, c2 + 1
        float xr[2][2][KW];  // [stream][channel][tap]: raw rows of tokens u-3 .. u
        auto ld2 = [&](int st, int r, float* x) {
          const uint32_t wv = *reinterpret_cast<const uint32_t*>(raw + st * Lay::RAWS + r * D * 2 + c2 * 2);
          x[0] = __uint_as_float(wv << 16);
          x[1] = __uint_as_float(wv & 0xffff0000u);
        };
#pragma unroll
        for (int st = 0; st < 2; ++st)
#pragma unroll
          for (int i = 0; i < KW - 1; ++i) {
            float x[2];
            ld2(st, ub + i, x);
            xr[st][0][i] = x[0];
            xr[st][1][i] = x[1];
          }
        const int cbox = (c2 >> 5) * 16384 + ((c2 & 3) << 2), cch = (c2 & 31) >> 2;
#pragma unroll 4
        for (int e = 0; e < 16; ++e) {
          const int u = ub + e;
#pragma unroll
          for (int st = 0; st < 2; ++st) {
            float x[2];
            ld2(st, u + KW - 1, x);
            float y[2];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              xr[st][cc][KW - 1] = x[cc];
              const float a = wq[st][cc][0] * xr[st][cc][0] + wq[st][cc][1] * xr[st][cc][1] +
                              wq[st][cc][2] * xr[st][cc][2] + wq[st][cc][3] * xr[st][cc][3];
              y[cc] = u < n ? silu(a) : 0.f;
#pragma unroll
              for (int i = 0; i < KW - 1; ++i) xr[st][cc][i] = xr[st][cc][i + 1];
            }
            const int r = st * C + u;
            *reinterpret_cast<float2*>(qk + cbox + r * 128 + ((cch ^ (r & 7)) << 4)) = make_float2(y[0], y[1]);
          }
        }
      }
      role_sync(1, NP);
      // ---- P5: next chunk's loads (the raw buffer is free); L2 norm of the 128 rows ----
      if (nsi < seg_end) issue_loads(nsi, nc0);
      // 8 threads per row, one 16-byte chunk of each of the 4 column boxes: the 8 lanes of
      // a 16-byte access phase then touch 8 different chunks of one box row (all 32 banks).
      // A thread's 4 rows (r, r + 32, r + 64, r + 96) are processed two at a time.
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int l8 = tid & 7, r0 = (tid >> 3) + 64 * half;
        float4 xv[2][4];
        float ss[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = r0 + 32 * i;
          const unsigned char* base = qk + r * 128 + ((l8 ^ (r & 7)) << 4);
          ss[i] = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            xv[i][q] = *reinterpret_cast<const float4*>(base + q * 16384);
            ss[i] += xv[i][q].x * xv[i][q].x + xv[i][q].y * xv[i][q].y + xv[i][q].z * xv[i][q].z + xv[i][q].w * xv[i][q].w;
          }
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], 1);
          ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], 2);
          ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], 4);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = r0 + 32 * i;
          unsigned char* base = qk + r * 128 + ((l8 ^ (r & 7)) << 4);
          const float inv = rsqrtf_(ss[i] + 1e-6f);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(base + q * 16384) =
                make_uint4(tf32_bits(xv[i][q].x * inv), tf32_bits(xv[i][q].y * inv), tf32_bits(xv[i][q].z * inv),
                           tf32_bits(xv[i][q].w * inv));
        }
      }
      tc::fence_proxy_async_smem();
      role_sync(1, NP);
      // ---- P6: [Q; K] K^T on the tensor cores; meanwhile diag(Gamma_last) K transposed
      //      (B operand of the state update) and (eta e^G K)^T (A operand of W^T) -------
      if (tid == 0) {
        tc::tc_fence_after();
        constexpr uint32_t id1 = tc::idesc_tf32(128, 64, 0, 0);
        const uint64_t dq = tc::sdesc_sw128(qk_a, 16, 1024), dk = tc::sdesc_sw128(qk_a + C * 128, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 8; ++ks) {
          const uint64_t off = static_cast<uint64_t>((ks >> 2) * 1024 + (ks & 3) * 2);
          tc::mma_tf32_ss(tmem + T_M1, dq + off, dk + off, id1, ks > 0);
        }
        tc::mma_commit(&bars[B_M1]);
      }
      // P and diag(Gamma_last) K^T are read by the chain's products of chunk k-1, and the
      // K^T tile then stages that chunk's output rows until the chain has written them out
      if (k >= 1 && !(ok = pwait(B_OUT, (k - 1) & 1))) break;
      {
        uint32_t kv4[32];
        float glv[32];
        ld32f(GL + u0, glv);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int t = u0 + e;
          const float kv = *reinterpret_cast<const float*>(qk + swz(128, C + t, ch));
          kv4[e] = tf32_bits(glv[e] * kv);
        }
        unsigned char* row = kt + hf * 16384 + ch * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(row + ((q ^ (ch & 7)) << 4)) =
              make_uint4(kv4[4 * q], kv4[4 * q + 1], kv4[4 * q + 2], kv4[4 * q + 3]);
      }
      // ---- P7: P (q rows) and A (k rows) from [Q; K] K^T -----------------------------
      if (!(ok = pwait(B_M1, k & 1))) break;
      tc::tc_fence_after();
      {
        uint32_t v32[32];
        tc::tmem_ld32(tmem + T_M1 + u0 + lb, v32);
        tc::tmem_wait_ld();
        const int t = ch < C ? ch : ch - C;
        const float gt = G[t] * kLog2e, et = ETA[t], egt = EG[t];
        // Gamma_ts = e^{G_t} e^{-G_s} while e^{-G} stays finite (G decreases along the
        // chunk), else 2^{(G_t - G_s) log2 e} per element
        const bool prod = G[C - 1] > -80.f;
        float vals[32];
        if (prod) {
          ld32f(IG + u0, vals);
#pragma unroll
          for (int e = 0; e < 32; ++e) vals[e] *= egt;
        } else {
          ld32f(G + u0, vals);
#pragma unroll
          for (int e = 0; e < 32; ++e) vals[e] = ex2f(gt - vals[e] * kLog2e);
        }
        // vals = Gamma_{t, u0+e}; masked and scaled by the products
        const float scale = ch < C ? 1.f : et;
        const int lim = ch < C ? t : t - 1;  // P keeps s <= t, A keeps s < t
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int s = u0 + e;
          vals[e] = s <= lim ? scale * vals[e] * __uint_as_float(v32[e]) : 0.f;
        }
        if (ch < C) {
          unsigned char* row = pb + hf * 8192 + t * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(row + ((q ^ (t & 7)) << 4)) =
                make_uint4(tf32_bits(vals[4 * q]), tf32_bits(vals[4 * q + 1]), tf32_bits(vals[4 * q + 2]),
                           tf32_bits(vals[4 * q + 3]));
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(&am[t * LDC + u0 + 4 * q]) =
                make_float4(vals[4 * q], vals[4 * q + 1], vals[4 * q + 2], vals[4 * q + 3]);
        }
      }
      tc::tc_fence_before();
      role_sync(1, NP);
      tc::tc_fence_after();
      // (eta e^G K)^T into the TMEM columns of Q K^T, now read by everyone
      {
        uint32_t aw[32];
        float etv[32], egv[32];
        ld32f(ETA + u0, etv);
        ld32f(EG + u0, egv);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int t = u0 + e;
          aw[e] = tf32_bits(etv[e] * egv[e] * *reinterpret_cast<const float*>(qk + swz(128, C + t, ch)));
        }
        tc::tmem_st32(tmem + T_M1 + u0 + lb, aw);
      }
      // ---- P8: T = (I + A)^{-1} (fp32): diagonal 16x16 blocks, then the others; each
      //      finished block also goes (rounded) into the B-operand tile --------------
      if (tid < 64) {
        const int bi = tid >> 4, c = tid & 15, base = bi * 16;
        float xv[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float a0 = (r == c) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
          for (int m = 0; m < r; m += 2) {
            a0 -= am[(base + r) * LDC + base + m] * xv[m];
            if (m + 1 < r) a1 -= am[(base + r) * LDC + base + m + 1] * xv[m + 1];
          }
          xv[r] = r < c ? 0.f : a0 + a1;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          tm[(base + r) * LDC + base + c] = xv[r];
          *reinterpret_cast<uint32_t*>(tb + swz(64, base + r, base + c)) = tf32_bits(xv[r]);
        }
      }
      role_sync(1, NP);
      // Off-diagonal blocks of T in two levels (T_ij = -T_ii A_ij T_jj for a 2 x 2 block
      // lower-triangular matrix): first the 16 x 16 blocks (1,0) and (3,2), then the 32 x 32
      // block T_BA = -T_BB (A_BA T_AA) with T_AA, T_BB the two 32 x 32 diagonal blocks.
      // Thread = (row, four columns): one float4 of T per term, so each shared-memory load
      // feeds four products.  T's upper blocks (0,1) and (2,3) hold zeros (set at the
      // start), so the sums run over whole blocks; Y = A_BA T_AA goes to T's unused
      // upper-right quarter.
      auto dot16 = [&](const float* arow, const float* bcol, int ldb, float4& acc) {
#pragma unroll
        for (int m4 = 0; m4 < 16; m4 += 4) {
          const float4 a = *reinterpret_cast<const float4*>(arow + m4);
          const float av4[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 t4 = *reinterpret_cast<const float4*>(bcol + (m4 + i) * ldb);
            acc.x += av4[i] * t4.x;
            acc.y += av4[i] * t4.y;
            acc.z += av4[i] * t4.z;
            acc.w += av4[i] * t4.w;
          }
        }
      };
      auto put_t = [&](int row, int col4, const float4& acc) {  // T(row, col4..+3) = -acc
        const float v4[4] = {-acc.x, -acc.y, -acc.z, -acc.w};
        *reinterpret_cast<float4*>(tm + row * LDC + col4) = make_float4(v4[0], v4[1], v4[2], v4[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) *reinterpret_cast<uint32_t*>(tb + swz(64, row, col4 + i)) = tf32_bits(v4[i]);
      };
      {
        const int pr = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
        const int bi = 2 * pr + 1, bj = 2 * pr;
        if (tid < 128) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          dot16(am + (bi * 16 + r) * LDC + bj * 16, tm + (bj * 16) * LDC + bj * 16 + c4, LDC, acc);
          *reinterpret_cast<float4*>(xs + (pr << 8) + r * 16 + c4) = acc;
        }
        role_sync(1, NP);
        if (tid < 128) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          dot16(tm + (bi * 16 + r) * LDC + bi * 16, xs + (pr << 8) + c4, 16, acc);
          put_t(bi * 16 + r, bj * 16 + c4, acc);
        }
        role_sync(1, NP);
      }
      {
        const int i = tid >> 3, c4 = (tid & 7) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        dot16(am + (32 + i) * LDC, tm + c4, LDC, acc);
        dot16(am + (32 + i) * LDC + 16, tm + 16 * LDC + c4, LDC, acc);
        *reinterpret_cast<float4*>(tm + i * LDC + 32 + c4) = acc;
        role_sync(1, NP);
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
        dot16(tm + (32 + i) * LDC + 32, tm + 32 + c4, LDC, acc);
        dot16(tm + (32 + i) * LDC + 48, tm + 16 * LDC + 32 + c4, LDC, acc);
        put_t(32 + i, c4, acc);
        role_sync(1, NP);
      }
      // ---- P9: W^T into the X columns of this slot (free once the chain has written out
      //      chunk k-2's rows) and U~^T into its U columns ---------------------------------
      if (k >= 2 && !(ok = pwait(B_EPI0 + slot, ((k - 2) >> 1) & 1))) break;
      tc::tmem_wait_st();
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      role_sync(1, NP);
      if (tid == 0) {
        tc::tc_fence_after();
        constexpr uint32_t id4 = tc::idesc_tf32(128, 64, 0, 0);
        for (int ks = 0; ks < C / 8; ++ks) {
          const uint64_t bd = tc::sdesc_sw128(tb_a + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
          tc::mma_tf32_ts(tmem + t_x(slot), tmem + T_M1 + ks * 8, bd, id4, ks > 0);
          tc::mma_tf32_ts(tmem + t_u(slot), tmem + T_AV + ks * 8, bd, id4, ks > 0);
        }
        tc::mma_commit(&bars[B_MW]);
      }
      // ---- P10: -W (rounded) replaces K in the operand tile -------------------------
      if (!(ok = pwait(B_MW, k & 1))) break;
      tc::tc_fence_after();
      {
        uint32_t v32[32];
        tc::tmem_ld32(tmem + t_x(slot) + u0 + lb, v32);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          *reinterpret_cast<uint32_t*>(qk + swz(128, C + u0 + e, ch)) = tf32_bits(-__uint_as_float(v32[e]));
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      role_sync(1, NP);
      if (tid == 0) tc::mbar_arrive(&bars[B_PREP]);
      ++k;
      si = nsi;
      c0 = nc0;
    }
    // drain: own MMAs, and a raw-row load still in flight after an abort (the last one
    // issued: its phase is the barrier's last)
    if (tid == 0) {
      tc::mma_commit(&bars[B_FINP]);
      tc::mbar_drain(&bars[B_FINP], 0);
      if (!ok && raw_issued > 0) tc::mbar_drain(&bars[B_RAW], (raw_issued - 1) & 1);
    }
    asm volatile("cp.async.wait_group 0;\n" ::);
  } else {
    // ============================ state chain (128 threads) ============================
    const int ct = tid - NP;
    const int v = q4 * 32 + lane;  // row of S (v index) = TMEM lane
    auto cwait = [&](int b, uint32_t par) -> bool {
      return role_and(2, NCH, tc::mbar_wait(&bars[b], par, abort, p.wait_ns));
    };
    // S <- a state from global memory (row v), or zero
    auto load_state = [&](const float* src) {
#pragma unroll
      for (int cb = 0; cb < D; cb += 32) {
        uint32_t v32[32];
        if (src) {
          const float4* s4 = reinterpret_cast<const float4*>(src + state_base + static_cast<int64_t>(v) * D + cb);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 f = s4[q];
            v32[4 * q] = __float_as_uint(f.x);
            v32[4 * q + 1] = __float_as_uint(f.y);
            v32[4 * q + 2] = __float_as_uint(f.z);
            v32[4 * q + 3] = __float_as_uint(f.w);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v32[e] = 0u;
        }
        tc::tmem_st32(tmem + T_S + cb + lb, v32);
      }
      tc::tmem_wait_st();
    };
    if (!BRANCH) load_state(S0);
    bool ok = !p.stall || cwait(B_STALL, 0);  // FORK_TEST_STALL: runs out, nothing is issued
    int si = first_seg(seg_first), c0 = 0, k = 0;
    while (ok && si < seg_end) {
      const int start = seg_start(si), len = seg_len(si), pos0 = seg_pos0(si);
      const int n = min(C, len - c0);
      const int slot = k & 1;
      const float* G = gslot + slot * 5 * C;
      const float* EG = G + C;
      const bool need_state = !BRANCH || (c0 + C < len);
      // ---- C0: operands of chunk k ready; a question starts from its request's S_P ----
      if (!(ok = cwait(B_PREP, k & 1))) break;
      if (BRANCH && c0 == 0) load_state(S0);
      tc::tc_fence_before();
      role_sync(2, NCH);
      if (ct == 0) {
        tc::tc_fence_after();
        constexpr uint32_t ida = tc::idesc_tf32(128, 64, 0, 0);
        const uint64_t dq = tc::sdesc_sw128(qk_a, 16, 1024), dw = tc::sdesc_sw128(qk_a + C * 128, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 8; ++ks) {
          const uint64_t off = static_cast<uint64_t>((ks >> 2) * 1024 + (ks & 3) * 2);
          tc::mma_tf32_ts(tmem + t_u(slot), tmem + T_S + ks * 8, dw + off, ida, 1u);  // U~^T - S W^T
          tc::mma_tf32_ts(tmem + t_x(slot), tmem + T_S + ks * 8, dq + off, ida, ks > 0);  // S Q^T
        }
        tc::mma_commit(&bars[B_MA]);
      }
      // ---- C1: U^T to TF32, X scaled by e^G, checkpoint, S scaled by e^{G_last} ------
      if (!(ok = cwait(B_MA, k & 1))) break;
      tc::tc_fence_after();
      {
        uint32_t v32[32];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          tc::tmem_ld32(tmem + t_u(slot) + q * 32 + lb, v32);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v32[e] = tf32_bits(__uint_as_float(v32[e]));
          tc::tmem_st32(tmem + t_u(slot) + q * 32 + lb, v32);
          tc::tmem_ld32(tmem + t_x(slot) + q * 32 + lb, v32);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v32[e] = __float_as_uint(__uint_as_float(v32[e]) * EG[q * 32 + e]);
          tc::tmem_st32(tmem + t_x(slot) + q * 32 + lb, v32);
        }
      }
      if (!BRANCH && ck >= 0 && p.S_ckpt) {
        // state after r of this chunk's tokens (rare): e^{G_{r-1}} S0 + sum_{s<r}
        // e^{G_{r-1} - G_s} u_s k_s^T, with k_s = (Gamma_last-scaled copy) / Gamma_last,s
        const int r_ck = ck - pos0 - c0;
        if (r_ck >= 1 && r_ck <= n) {
          tc::tmem_wait_st();
          uint32_t ua[32], ub[32], s32[32];
          tc::tmem_ld32(tmem + t_u(slot) + lb, ua);
          tc::tmem_ld32(tmem + t_u(slot) + 32 + lb, ub);
          tc::tmem_wait_ld();
          const float gr = G[r_ck - 1], f = expf(gr - G[C - 1]);
          for (int cb = 0; cb < D; cb += 32) {
            tc::tmem_ld32(tmem + T_S + cb + lb, s32);
            tc::tmem_wait_ld();
            float acc[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[e] = expf(gr) * __uint_as_float(s32[e]);
            for (int s = 0; s < r_ck; ++s) {
              const float us = __uint_as_float(s < 32 ? ua[s & 31] : ub[s & 31]) * f;
#pragma unroll
              for (int e = 0; e < 32; ++e) acc[e] += us * *reinterpret_cast<const float*>(kt + swz(128, cb + e, s));
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) p.S_ckpt[state_base + static_cast<int64_t>(v) * D + cb + e] = acc[e];
          }
        }
      }
      if (need_state) {
        const float egl = EG[C - 1];
        uint32_t v32[32];
#pragma unroll
        for (int cb = 0; cb < D; cb += 32) {
          tc::tmem_ld32(tmem + T_S + cb + lb, v32);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v32[e] = __float_as_uint(__uint_as_float(v32[e]) * egl);
          tc::tmem_st32(tmem + T_S + cb + lb, v32);
        }
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      role_sync(2, NCH);
      // ---- C2: O^T += U^T P^T and S += U^T diag(Gamma_last) K ---------------------------
      if (ct == 0) {
        tc::tc_fence_after();
        constexpr uint32_t id5 = tc::idesc_tf32(128, 64, 0, 0);
        constexpr uint32_t id6 = tc::idesc_tf32(128, 128, 0, 0);
        for (int ks = 0; ks < C / 8; ++ks)
          tc::mma_tf32_ts(tmem + t_x(slot), tmem + t_u(slot) + ks * 8,
                          tc::sdesc_sw128(pb_a + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), id5, 1u);
        if (need_state)
          for (int ks = 0; ks < C / 8; ++ks)
            tc::mma_tf32_ts(tmem + T_S, tmem + t_u(slot) + ks * 8,
                            tc::sdesc_sw128(kt_a + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024), id6, 1u);
        tc::mma_commit(&bars[B_MB]);
      }
      // ---- C3: output rows.  Thread v holds column v of the chunk's 64 x 128 output; the
      //      columns are staged as bf16 rows (token-major, 256 bytes each) in the K^T tile,
      //      free now that the products of this chunk are complete, then written out as
      //      coalesced 16-byte stores.  Lane pairs swap values so that each shared-memory
      //      store carries two neighbouring columns of one token; odd rows are rotated by
      //      64 bytes so that the two tokens of one store instruction use different banks.
      if (!(ok = cwait(B_MB, k & 1))) break;
      tc::tc_fence_after();
      {
        const bool odd = lane & 1;
        const int v0 = v & ~1;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t v32[32];
          tc::tmem_ld32(tmem + t_x(slot) + q * 32 + lb, v32);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            // even lane: (token t, columns v, v+1); odd lane: (token t+1, columns v-1, v)
            const float mine_t = __uint_as_float(v32[e]), mine_t1 = __uint_as_float(v32[e + 1]);
            const float other = __shfl_xor_sync(0xffffffffu, odd ? mine_t : mine_t1, 1);
            const int t = q * 32 + e + (odd ? 1 : 0);
            const __nv_bfloat162 pr = odd ? __floats2bfloat162_rn(other, mine_t1) : __floats2bfloat162_rn(mine_t, other);
            *reinterpret_cast<__nv_bfloat162*>(kt + t * (D * 2) + ((v0 * 2 + (t & 1) * 64) & (D * 2 - 1))) = pr;
          }
        }
      }
      role_sync(2, NCH);
      {
        const int cq = ct & 15;  // 16-byte piece of a 256-byte row
#pragma unroll
        for (int pass = 0; pass < C / 8; ++pass) {
          const int t = pass * 8 + (ct >> 4);
          if (t < n) {
            const uint4 val = *reinterpret_cast<const uint4*>(kt + t * (D * 2) + ((cq * 16 + (t & 1) * 64) & (D * 2 - 1)));
            *reinterpret_cast<uint4*>(p.o + (static_cast<int64_t>(start + c0 + t) * H + h) * D + cq * 8) = val;
          }
        }
      }
      tc::mbar_arrive(&bars[B_OUT]);
      tc::tc_fence_before();
      tc::mbar_arrive(&bars[B_EPI0 + slot]);
      ++k;
      c0 += C;
      if (c0 >= len) {
        si = first_seg(si + 1);
        c0 = 0;
      }
    }
    if (ok && !BRANCH) {
      // S_P from TMEM
      uint32_t v32[32];
#pragma unroll
      for (int cb = 0; cb < D; cb += 32) {
        tc::tmem_ld32(tmem + T_S + cb + lb, v32);
        tc::tmem_wait_ld();
        float4* dst = reinterpret_cast<float4*>(p.S_P + state_base + static_cast<int64_t>(v) * D + cb);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_float4(__uint_as_float(v32[4 * q]), __uint_as_float(v32[4 * q + 1]),
                               __uint_as_float(v32[4 * q + 2]), __uint_as_float(v32[4 * q + 3]));
      }
    }
    if (ct == 0) {
      tc::mma_commit(&bars[B_FINC]);
      tc::mbar_drain(&bars[B_FINC], 0);
    }
  }

  if (!BRANCH && !*abort) {
    // conv windows: raw q, k, v inputs of the trunk's last K-1 positions (and of the K-1
    // positions before a checkpoint), zero before position 0 of the request
    const int start = meta[L.seg_start + j], len = meta[L.seg_len + j], pos0 = meta[L.seg_pos0 + j];
    auto raw_in = [&](int o_seg, int s, int c) -> uint16_t {
      const uint16_t* src = s == 0 ? p.q : (s == 1 ? p.k : p.v);
      if (o_seg >= 0) return src[(static_cast<int64_t>(start + o_seg) * H + h) * D + c];
      const int r = KW - 1 + o_seg;
      if (r < 0 || hist == nullptr) return 0;
      return hist[((static_cast<int64_t>(j * (KW - 1) + r) * 3 + s) * H + h) * D + c];
    };
    for (int e = tid; e < (KW - 1) * 3 * D; e += NT) {
      const int i = e / (3 * D), s = (e / D) % 3, c = e % D;
      const int64_t dst = ((static_cast<int64_t>(j * (KW - 1) + i) * 3 + s) * H + h) * D + c;
      p.conv_win[dst] = raw_in(len - (KW - 1) + i, s, c);
      if (ck >= 0 && p.conv_ckpt) p.conv_ckpt[dst] = raw_in(ck - pos0 - (KW - 1) + i, s, c);
    }
  }
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
  alignas(128) CUtensorMap maps[3];
  const uint16_t* src[3] = {p.q, p.k, p.v};
  for (int i = 0; i < 3; ++i)
    if (!encode_map_3d(&maps[i], src[i], D, p.H, p.L.T_cap, D, 1, HR, false)) return FORK_ECUDA;
  dim3 grid(grid_x, p.H);
  if (branch) {
    if (cuda_rc(cudaFuncSetAttribute(gdn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM)) !=
        FORK_OK)
      return FORK_ECUDA;
    gdn_tc_kernel<true><<<grid, NT, Lay::SMEM, s>>>(maps[0], maps[1], maps[2], p);
  } else {
    if (cuda_rc(cudaFuncSetAttribute(gdn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM)) !=
        FORK_OK)
      return FORK_ECUDA;
    gdn_tc_kernel<false><<<grid, NT, Lay::SMEM, s>>>(maps[0], maps[1], maps[2], p);
  }
  return cuda_rc(cudaGetLastError());
}

}  // namespace fork
