// Two-call forked Gated DeltaNet on the 5th-generation tensor cores (tcgen05, fp16 operands).
//
// Gated delta rule of the rainbus summary "前置知识", in the chunked form that the
// DFlash-TfM summary ("GDN을 위한 롤백 없는 트리 검증") solves with a Gram matrix and a
// triangular solve.  For a chunk of C = 64 tokens with start state S0 (d_v x d_k),
// G_t = sum_{s<=t} log a_s, Gamma_ts = exp(G_t - G_s):
//   A_ts = eta_t Gamma_ts k_t.k_s (s < t),  T = (I + A)^{-1}
//   W = T diag(eta e^G) K,  U~ = T diag(eta) V        (independent of S0)
//   U = U~ - W S0^T
//   O = diag(e^G) Q S0^T + (tril(Gamma) * Q K^T) U
//   S = e^{G_last} S0 + U^T diag(Gamma_last) K.
// The L2 normalisation of q and k is never applied to a tile: with Y the conv + SiLU
// rows and n_t = (sum_c Y_tc^2 + 1e-6)^(-1/2), K = diag(n_k) Y_k and Q = diag(n_q) Y_q,
// so every product above takes the norms as row or column factors of a small matrix
// (P, A, T diag(.), the output scale, the state-update scale) and the tensor cores read
// Y itself.
//
// One CTA = one trunk (call 1) or a group of up to kQG questions of one request
// (call 2) x one head; d = 128.  A node of a token forest runs as a trunk that starts
// from its parent's end state (the state index of the trunk's segment).  16 warps in three roles that work on consecutive chunks
// (two slots of row tiles, so the roles overlap):
//   warps 0-3   conv of chunk k+1 for q and k: raw rows by TMA (the chunk and the three
//               rows before it, 128-byte swizzled; the next chunk's rows are requested as
//               soon as this chunk's are read), thread = (8 channels, 8 tokens): causal
//               conv + SiLU over a sliding window of unpacked rows with the weights in
//               registers, fp16 rows into the operand tiles, the L2 norms from sums of
//               squares reduced over a half warp; the raw gates by cp.async.
//   warps 4-11  solve of chunk k+1 (everything above the line "U = ..."): the gates
//               (first warp, while the tensor cores run); [Y_q; Y_k] Y_k^T on the tensor
//               cores -> P (fp16) and A (fp32); T = (I + A)^{-1} in fp32 (16x16 diagonal
//               blocks by forward substitution, the rest in two levels); T diag(eta e^G
//               n_k) and T diag(eta) as fp16 tiles; W^T = Y_k^T (T diag(eta e^G n_k))^T and
//               U~^T = Y_v^T (T diag(eta))^T on the tensor cores; -W as an fp16 tile.
//   warps 12-15 state chain of chunk k (thread = TMEM lane = row v of S): U^T = U~^T -
//               S W^T and X = S Y_q^T (A operand: an fp16 copy of S in tensor memory);
//               U^T to fp16 twice (plain, and scaled by Gamma_last n_k for the update); X
//               scaled by e^G n_q; S by e^{G_last}; then O^T = X + U^T P^T and
//               S += (U^T diag(Gamma_last n_k)) Y_k; output rows; the fp16 copy of S.
//               Between its chunks the chain makes Y_v of chunk k+1 (the same conv as
//               above, on its own raw rows), which the solve group's U~ product waits for.
// S (128 x 128 fp32) stays in tensor memory for the whole segment.  Operands are fp16
// (10-bit mantissa, as TF32; the values stay far inside the fp16 range), products
// accumulate in fp32, T is formed in fp32.  Every wait is bounded and agreed by the
// threads of its role.
#include <cuda_fp16.h>

#include "fork_attn.cuh"
#include "fork_gdn.cuh"
#include "tc_ptx.cuh"

namespace fork {

namespace {
constexpr int D = 128;
constexpr int C = 64;
constexpr int NCV = 128;       // conv group (4 warps)
constexpr int NSV = 256;       // solve group (8 warps)
constexpr int NCH = 128;       // chain threads (4 warps)
constexpr int NT = NCV + NSV + NCH;
constexpr int KW = 4;
constexpr int HR = C + KW - 1;  // raw rows staged per chunk
constexpr int LDC = C + 4;      // plain 64-wide fp32 tiles
constexpr int kQG = 4;          // questions per CTA in the branch call (8 measured the same)
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S (fp32), its fp16 copy, two U slots, X, the prep's product, two scaled
// fp16 copies of U^T
constexpr uint32_t T_S = 0, T_S16 = 128, T_X = 320, T_M1 = 384;
__device__ __forceinline__ uint32_t t_u(int slot) { return 192u + 64u * slot; }
// U^T diag(Gamma_last n_k) as fp16 pairs (A operand of the state update), per slot
__device__ __forceinline__ uint32_t t_ug(int slot) { return 448u + 32u * slot; }

struct Lay {
  static constexpr int RAWH = 9216;               // one 64-channel half of a stream's raw rows (HR used)
  static constexpr int RAW = 0;                   // [3 streams][2 halves] bf16, 128-byte swizzled
  static constexpr int YTS = 32768;               // one slot: [2 boxes][Y_q rows 0-63; Y_k rows 64-127][128 B]
  static constexpr int YT = RAW + 6 * RAWH;       // [2 slots]
  static constexpr int YV = YT + 2 * YTS;         // Y_v [2 boxes][64 rows][128 B]
  static constexpr int WT = YV + 16384;           // -W  [2 boxes][64 rows][128 B]
  static constexpr int PB = WT + 16384;           // P   [2 slots][64 rows][128 B]; output staging
  static constexpr int TP = PB + 2 * 8192;        // T diag(eta e^G n_k) [64][128 B]
  static constexpr int TPP = TP + 8192;           // T diag(eta)         [64][128 B]
  static constexpr int AM = TPP + 8192;           // A fp32 [64][LDC]
  static constexpr int TM = AM + C * LDC * 4;     // T fp32 [64][LDC]
  static constexpr int GA = TM + C * LDC * 4;     // raw alpha, eta per slot [2][2][64]
  static constexpr int GS = GA + 2 * 2 * C * 4;   // per slot [G, EG, GL, ETA, IG, NQ, NK][64]
  static constexpr int SEG = GS + 2 * 7 * C * 4;  // this CTA's segments: start, len, pos0
  static constexpr int BAR = SEG + (3 * kQG * 4 + 63) / 64 * 64;
  static constexpr int BYTES = BAR + 256;
  static constexpr int SMEM = BYTES + 1024;
};
static_assert(Lay::SMEM <= 232448, "shared memory budget");
static_assert(kQG * 3 <= NT, "segment table filled by one thread per entry");
static_assert(Lay::YT % 1024 == 0 && Lay::YV % 1024 == 0 && Lay::WT % 1024 == 0 && Lay::PB % 1024 == 0 &&
                  Lay::TP % 1024 == 0 && Lay::TPP % 1024 == 0 && Lay::RAWH % 1024 == 0,
              "128-byte-swizzled tiles start on 1024-byte boundaries");
static_assert(HR * 128 <= Lay::RAWH, "raw rows");

enum { B_RAWQK = 0, B_RAWV, B_CONV, B_M1, B_MW, B_PREP, B_MA, B_MB, B_EPI0, B_EPI1, B_PF0, B_PF1, B_FINP, B_FINC, B_STALL,
       B_GATE, B_YV, B_N };
enum { G_G = 0, G_EG, G_GL, G_ETA, G_IG, G_NQ, G_NK };

// SFU approximations: 2^x, 1/sqrt(x) (relative error ~2^-22), tanh (~2^-11)
__device__ __forceinline__ float tanhf_(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rsqrtf_(float x) {
  float y;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;
// SiLU(y) = y sigmoid(y) = y/2 + (y/2) tanh(y/2): one SFU operation.  The tanh error is
// relative to tanh(y/2), so the result keeps ~2^-11 relative precision wherever the conv
// outputs live (|y| of a few units), the precision of the fp16 operand it becomes.
__device__ __forceinline__ float silu(float y) {
  const float h = 0.5f * y;
  return fmaf(h, tanhf_(h), h);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// byte offset of 16-byte chunk j of row r in a 128-byte-swizzled box of 128-byte rows
__device__ __forceinline__ int sw(int r, int j) { return r * 128 + ((j ^ (r & 7)) << 4); }
__device__ __forceinline__ void cp_async4(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(tc::smem_u32(dst)), "l"(src),
               "r"(valid ? 4 : 0));
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
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
// the i-th 32-bit word of a 16-byte vector (i a compile-time constant after unrolling)
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
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
    // a round's trunks, or the segments [seg_base, seg_base + n_segs) of a forest level
    if (x >= (p.n_segs >= 0 ? p.n_segs : R)) return;
    j = p.seg_base + x;
    if (j >= R) return;
    seg_first = j;
    seg_end = j + 1;
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
  // index of the start state and conv window: the request's own (a question reads S_P[j], a
  // resumed trunk its init_state[j]), or a forest node's parent's (its segment's state index)
  const int in_idx = BRANCH ? j : meta[L.seg_state_idx + j];
  if (resumed && (in_idx < 0 || in_idx >= R)) {
    if (tid == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_BAD_PREFIX);
    return;
  }
  const uint16_t* hist = (BRANCH || resumed) ? p.hist_in : nullptr;
  const float* S0 = (BRANCH || resumed) ? p.state_in : nullptr;
  const int64_t state_base = (static_cast<int64_t>(j) * H + h) * D * D;  // outputs
  const int64_t in_base = (static_cast<int64_t>(in_idx) * H + h) * D * D;

  unsigned char* raw = sm + Lay::RAW;
  unsigned char* yv = sm + Lay::YV;
  unsigned char* wt = sm + Lay::WT;
  unsigned char* tp = sm + Lay::TP;
  unsigned char* tpp = sm + Lay::TPP;
  float* am = reinterpret_cast<float*>(sm + Lay::AM);
  float* tm = reinterpret_cast<float*>(sm + Lay::TM);
  float* ga = reinterpret_cast<float*>(sm + Lay::GA);  // [slot][alpha, eta][64]
  int* segt = reinterpret_cast<int*>(sm + Lay::SEG);  // [kQG][3], read instead of the metadata
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::BAR + B_N * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + Lay::BAR + B_N * 8 + 8);
  auto yt = [&](int slot) { return sm + Lay::YT + slot * Lay::YTS; };
  auto pbt = [&](int slot) { return sm + Lay::PB + slot * 8192; };
  auto gate = [&](int slot, int a) { return reinterpret_cast<float*>(sm + Lay::GS) + (slot * 7 + a) * C; };

  if (tid == 0) {
    // B_STALL is completed by nothing (FORK_TEST_STALL)
    for (int b = 0; b < B_N; ++b)
      tc::mbar_init(&bars[b], (b == B_EPI0 || b == B_EPI1 || b == B_PF0 || b == B_PF1) ? NCH : b == B_GATE ? 32 : 1);
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
    for (int e = tid; e < D * D; e += NT) p.S_ckpt[state_base + e] = S0 ? S0[in_base + e] : 0.f;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
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

  // ---- raw rows and the causal conv, shared by the conv group (q, k) and the chain (v) ----
  const CUtensorMap* maps[3] = {&qmap, &kmap, &vmap};
  // raw rows (the chunk and the three before it; rows outside the tensor read as zero) of
  // streams [s_lo, s_hi) of a chunk, on barrier b (one thread)
  auto issue_rows = [&](int s, int cc, int s_lo, int s_hi, int b) {
    tc::fence_proxy_async_smem();  // the rows were last read (and patched) by threads
    tc::mbar_expect_tx(&bars[b], (s_hi - s_lo) * 2 * HR * 128);
    for (int s3 = s_lo; s3 < s_hi; ++s3)
#pragma unroll
      for (int half = 0; half < 2; ++half)
        tc::tma_load_3d(raw + (s3 * 2 + half) * Lay::RAWH, maps[s3], &bars[b], half * 64, h, seg_start(s) + cc - (KW - 1));
  };
  // history rows of a segment start for streams [s_lo, s_hi), by the 128 threads r of a
  // role: raw inputs before the segment (the request's conv window for a question or a
  // resumed trunk, else zero)
  auto patch_history = [&](int r, int s_lo, int s_hi) {
    for (int e = r; e < (s_hi - s_lo) * (KW - 1) * D; e += 128) {
      const int s3 = s_lo + e / ((KW - 1) * D), i = (e / D) % (KW - 1), c = e % D;
      const uint16_t hv =
          hist ? hist[((static_cast<int64_t>(in_idx * (KW - 1) + i) * 3 + s3) * H + h) * D + c] : uint16_t(0);
      *reinterpret_cast<uint16_t*>(raw + (s3 * 2 + (c >> 6)) * Lay::RAWH + sw(i, (c & 63) >> 3) + (c & 7) * 2) = hv;
    }
  };
  // conv + SiLU of stream st over a chunk with n valid tokens, by the 128 threads r of a
  // role: thread = 8-channel group cg (channels 8cg..8cg+7) x block of 8 tokens tb (the 16
  // lanes of a half warp hold the 128 channels of the same 8 tokens), a sliding window of
  // raw rows (positions u-3..u for token u), each row unpacked once; fp16 rows into box
  // (cg / 8) of `tile` (boxes of box_bytes, rows row0 + u); for q and k the norm
  // (sum_c y^2 + 1e-6)^(-1/2) of each token into nrm, from sums of squares over the 16
  // lanes of a token block
  auto conv_stream = [&](int r, int st, int n, unsigned char* tile, int box_bytes, int row0, float* nrm) {
    const int cg = r & 15, tb = r >> 4;
    const float4* cw4 = reinterpret_cast<const float4*>(p.conv_w) + ((static_cast<int64_t>(st) * H + h) * D + 8 * cg);
    const unsigned char* rb = raw + (st * 2 + (cg >> 3)) * Lay::RAWH;
    const int jc = cg & 7;
    unsigned char* dst = tile + (cg >> 3) * box_bytes;
    const int u0 = tb * 8;
    float cw[8][KW];  // the group's conv weights (8 channels x 4 taps), L1-resident
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float4 w = __ldg(cw4 + e);
      cw[e][0] = w.x;
      cw[e][1] = w.y;
      cw[e][2] = w.z;
      cw[e][3] = w.w;
    }
    float xw[KW][8];  // unpacked raw rows u-3..u of the 8 channels
    auto unpack = [&](int row, float* x) {
      const uint4 r4 = *reinterpret_cast<const uint4*>(rb + sw(row, jc));
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t word = word_of(r4, q);
        x[2 * q] = bf_lo(word);
        x[2 * q + 1] = bf_hi(word);
      }
    };
#pragma unroll
    for (int i = 0; i < KW - 1; ++i) unpack(u0 + i, xw[i + 1]);
    float ssum[8];
#pragma unroll
    for (int uu = 0; uu < 8; ++uu) {
      const int u = u0 + uu;
#pragma unroll
      for (int i = 0; i < KW - 1; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) xw[i][e] = xw[i + 1][e];
      unpack(u + KW - 1, xw[KW - 1]);  // position u
      float y[8];
      float sq = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float a = cw[e][0] * xw[0][e];
#pragma unroll
        for (int i = 1; i < KW; ++i) a = fmaf(cw[e][i], xw[i][e], a);
        y[e] = u < n ? silu(a) : 0.f;
        sq = fmaf(y[e], y[e], sq);
      }
      ssum[uu] = sq;
      *reinterpret_cast<uint4*>(dst + sw(row0 + u, jc)) =
          make_uint4(pack_h2(y[0], y[1]), pack_h2(y[2], y[3]), pack_h2(y[4], y[5]), pack_h2(y[6], y[7]));
    }
    if (nrm) {
#pragma unroll
      for (int uu = 0; uu < 8; ++uu) {
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) ssum[uu] += __shfl_xor_sync(0xffffffffu, ssum[uu], o);
      }
      if (cg < 8) {
        float sv = ssum[0];
#pragma unroll
        for (int uu = 1; uu < 8; ++uu)
          if (cg == uu) sv = ssum[uu];
        nrm[u0 + cg] = rsqrtf_(sv + 1e-6f);
      }
    }
  };

  if (warp < NCV / 32) {
    // ============================ conv group (128 threads): q, k ============================
    auto cvwait = [&](int b, uint32_t par) -> bool {
      return role_and(1, NCV, tc::mbar_wait(&bars[b], par, abort, p.wait_ns));
    };
    int qk_issued = 0;
    // the raw gates of a chunk into its staging slot (read by the solve group)
    auto issue_gates = [&](int s, int cc, int gslot) {
      const int st0 = seg_start(s), ln = seg_len(s);
      const int uu = tid & (C - 1);
      const bool valid = cc + uu < ln;
      const float* src = (tid < C ? p.alpha : p.eta) + (static_cast<int64_t>(st0 + (valid ? cc + uu : 0)) * H + h);
      cp_async4(ga + gslot * 2 * C + (tid < C ? 0 : C) + uu, src, valid);
      asm volatile("cp.async.commit_group;\n" ::);
    };
    if (tid == 0) {
      tc::prefetch_tmap(&qmap);
      tc::prefetch_tmap(&kmap);
    }
    bool ok = true;
    int si = first_seg(seg_first), c0 = 0, k = 0;
    if (si < seg_end) {
      if (tid == 0) issue_rows(si, 0, 0, 2, B_RAWQK);
      issue_gates(si, 0, 0);
      ++qk_issued;
    }
    while (ok && si < seg_end) {
      const int len = seg_len(si);
      const int n = min(C, len - c0);
      const int slot = k & 1;
      unsigned char* yts = yt(slot);
      int nsi = si, nc0 = c0 + C;
      if (nc0 >= len) {
        nsi = first_seg(si + 1);
        nc0 = 0;
      }
      // this chunk's q, k rows have landed; history rows of a segment start; the slot's tiles
      // are free once the chain's products of chunk k-2 are done
      if (!(ok = cvwait(B_RAWQK, (qk_issued - 1) & 1))) break;
      if (c0 == 0) patch_history(tid, 0, 2);
      if (k >= 2 && !(ok = cvwait(B_EPI0 + slot, ((k - 2) >> 1) & 1))) break;
      role_sync(1, NCV);
      conv_stream(tid, 0, n, yts, 16384, 0, gate(slot, G_NQ));
      conv_stream(tid, 1, n, yts, 16384, C, gate(slot, G_NK));
      // the q, k rows are read: next chunk's loads
      role_sync(1, NCV);
      if (nsi < seg_end) {
        if (tid == 0) issue_rows(nsi, nc0, 0, 2, B_RAWQK);
        ++qk_issued;
      }
      asm volatile("cp.async.wait_group 0;\n" ::);  // this chunk's gates are staged
      tc::fence_proxy_async_smem();
      role_sync(1, NCV);
      if (tid == 0) tc::mbar_arrive(&bars[B_CONV]);
      // next chunk's gates (its gate slot was read by the solve group for chunk k-1, done
      // before this chunk's conv could start)
      if (nsi < seg_end) issue_gates(nsi, nc0, (k + 1) & 1);
      ++k;
      si = nsi;
      c0 = nc0;
    }
    // drain: raw-row loads still in flight after an abort (the last ones issued: their
    // phases are the barrier's last)
    if (tid == 0 && !ok && qk_issued > 0) tc::mbar_drain(&bars[B_RAWQK], (qk_issued - 1) & 1);
    asm volatile("cp.async.wait_group 0;\n" ::);
  } else if (warp < (NCV + NSV) / 32) {
    // ============================ solve group (256 threads) ============================
    const int stid = tid - NCV;
    auto swait = [&](int b, uint32_t par) -> bool {
      return role_and(3, NSV, tc::mbar_wait(&bars[b], par, abort, p.wait_ns));
    };
    // blocks (0,1) and (2,3) of the fp32 T stay zero (the two-level products read them)
    for (int e = stid; e < C * C; e += NSV) {
      const int t = e >> 6, s = e & 63;
      if ((s >> 4) == (t >> 4) + 1 && (t >> 4) % 2 == 0) tm[t * LDC + s] = 0.f;
    }
    bool ok = true;
    int si = first_seg(seg_first), c0 = 0, k = 0;
    while (ok && si < seg_end) {
      const int len = seg_len(si);
      const int slot = k & 1;
      float* G = gate(slot, G_G);
      float* EG = gate(slot, G_EG);
      float* ETA = gate(slot, G_ETA);
      float* IG = gate(slot, G_IG);
      float* NQ = gate(slot, G_NQ);
      float* NK = gate(slot, G_NK);
      unsigned char* yts = yt(slot);
      unsigned char* pb = pbt(slot);
      // ---- S0: the conv group has produced this chunk's rows, norms and raw gates; [Y_q; Y_k]
      //      Y_k^T on the tensor cores --------------------------------------------------
      if (!(ok = swait(B_CONV, k & 1))) break;
      if (stid == 0) {
        tc::tc_fence_after();
        constexpr uint32_t id1 = tc::idesc_fp16(128, 64, 0, 0);
        const uint64_t da = tc::sdesc_sw128(tc::smem_u32(yts), 16, 1024);
        const uint64_t db = tc::sdesc_sw128(tc::smem_u32(yts + C * 128), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t off = static_cast<uint64_t>((ks >> 2) * (16384 / 16) + (ks & 3) * 2);
          tc::mma_bf16(tmem + T_M1, da + off, db + off, id1, ks > 0);
        }
        tc::mma_commit(&bars[B_M1]);
      }
      // ---- S1: P (q rows) and A (k rows) from [Y_q; Y_k] Y_k^T; the P tile of this slot is
      //      free once the chain has written out chunk k-2's rows (it stages them there)
      // gates of this chunk (first solve warp, while the product runs; SFU log and exp: the
      // cumulative log gate is off by at most ~3e-5 over a chunk, far below the fp16
      // rounding of the operands it scales).  The gate slot is free once the chain has
      // finished chunk k-2, which it signals after reading chunk k-1's gates: the gate
      // barrier is never two phases ahead of the chain's waits on it.
      bool gok = true;
      if (stid < 32) {
        if (k >= 2) gok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_PF0 + slot], ((k - 2) >> 1) & 1, abort, p.wait_ns));
        if (gok) {
          const float* gas = ga + slot * 2 * C;
          const int n = min(C, len - c0);
          const int a0 = 2 * lane, a1 = a0 + 1;
          const float l0 = a0 < n ? __logf(gas[a0]) : 0.f, l1 = a1 < n ? __logf(gas[a1]) : 0.f;
          float xx = l0 + l1;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, xx, o);
            if (lane >= o) xx += y;
          }
          const float g1 = xx, g0 = xx - l1;
          const float glast = __shfl_sync(0xffffffffu, xx, 31);
          float* GL = gate(slot, G_GL);
          *reinterpret_cast<float2*>(G + a0) = make_float2(g0, g1);
          *reinterpret_cast<float2*>(EG + a0) = make_float2(__expf(g0), __expf(g1));
          *reinterpret_cast<float2*>(GL + a0) = make_float2(__expf(glast - g0), __expf(glast - g1));
          *reinterpret_cast<float2*>(ETA + a0) = make_float2(a0 < n ? gas[C + a0] : 0.f, a1 < n ? gas[C + a1] : 0.f);
          // used only when no G of the chunk is below -80 (no overflow)
          *reinterpret_cast<float2*>(IG + a0) = make_float2(__expf(-g0), __expf(-g1));
          tc::mbar_arrive(&bars[B_GATE]);  // every lane: each releases its own stores
        }
      }
      if (!(ok = role_and(3, NSV, gok && tc::mbar_wait(&bars[B_M1], k & 1, abort, p.wait_ns)))) break;
      if (k >= 2 && !(ok = swait(B_PF0 + slot, ((k - 2) >> 1) & 1))) break;
      tc::tc_fence_after();
      {
        const int ch = (warp - NCV / 32) >> 2;  // column half
        const int r = q4 * 32 + lane;
        const int u0 = ch * 32;
        uint32_t v32[32];
        tc::tmem_ld32(tmem + T_M1 + u0 + lb, v32);
        tc::tmem_wait_ld();
        const int t = r < C ? r : r - C;
        const float gt = G[t] * kLog2e, egt = EG[t];
        // Gamma_ts = e^{G_t} e^{-G_s} while e^{-G} stays finite (G decreases along the
        // chunk), else 2^{(G_t - G_s) log2 e} per element.
        // P_ts = n_q,t n_k,s Gamma_ts (Y_q Y_k^T)_ts (s <= t);
        // A_ts = eta_t n_k,t n_k,s Gamma_ts (Y_k Y_k^T)_ts (s < t)
        const bool prod = G[C - 1] > -80.f;
        const float scale = r < C ? NQ[t] : ETA[t] * NK[t];
        const int lim = r < C ? t : t - 1;
        float vals[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 nk = *reinterpret_cast<const float4*>(NK + u0 + 4 * q);
          const float4 gg = *reinterpret_cast<const float4*>((prod ? IG : G) + u0 + 4 * q);
          const float nkv[4] = {nk.x, nk.y, nk.z, nk.w}, ggv[4] = {gg.x, gg.y, gg.z, gg.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = 4 * q + i, s2 = u0 + e;
            const float gam = prod ? egt * ggv[i] : ex2f(gt - ggv[i] * kLog2e);
            vals[e] = s2 <= lim ? scale * nkv[i] * gam * __uint_as_float(v32[e]) : 0.f;
          }
        }
        if (r < C) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(pb + sw(t, ch * 4 + q)) =
                make_uint4(pack_h2(vals[8 * q], vals[8 * q + 1]), pack_h2(vals[8 * q + 2], vals[8 * q + 3]),
                           pack_h2(vals[8 * q + 4], vals[8 * q + 5]), pack_h2(vals[8 * q + 6], vals[8 * q + 7]));
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(&am[t * LDC + u0 + 4 * q]) =
                make_float4(vals[4 * q], vals[4 * q + 1], vals[4 * q + 2], vals[4 * q + 3]);
        }
      }
      tc::tc_fence_before();
      role_sync(3, NSV);
      // ---- S2: T = (I + A)^{-1} (fp32): diagonal 16x16 blocks, then the others ----------
      if (stid < 64) {
        const int bi = stid >> 4, c = stid & 15, base = bi * 16;
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
        for (int r = 0; r < 16; ++r) tm[(base + r) * LDC + base + c] = xv[r];
      }
      role_sync(3, NSV);
      // Off-diagonal blocks of T in two levels (T_ij = -T_ii A_ij T_jj for a 2 x 2 block
      // lower-triangular matrix): first the 16 x 16 blocks (1,0) and (3,2), then the 32 x 32
      // block T_BA = -T_BB (A_BA T_AA) with T_AA, T_BB the two 32 x 32 diagonal blocks.
      // T's blocks (0,1) and (2,3) hold zeros, so the sums run over whole blocks; Y = A_BA T_AA
      // goes to T's unused upper-right quarter.  Each thread computes one row x 4 columns; the
      // 4-column groups of a row are read once per warp (broadcast).
      // rows[i] (+)= sum_k X[r_i][k] * Z[k][c4..c4+3], X and Z row-major with stride ld
      auto blk = [&](float4* acc, int nr, const float* x0, const float* z0, int kn) {
#pragma unroll 2
        for (int k4 = 0; k4 < kn; k4 += 4) {
          float4 xv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < nr) xv[i] = *reinterpret_cast<const float4*>(x0 + i * LDC + k4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const float4 z = *reinterpret_cast<const float4*>(z0 + (k4 + kk) * LDC);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (i < nr) {
                const float xs_ = kk == 0 ? xv[i].x : kk == 1 ? xv[i].y : kk == 2 ? xv[i].z : xv[i].w;
                acc[i].x = fmaf(xs_, z.x, acc[i].x);
                acc[i].y = fmaf(xs_, z.y, acc[i].y);
                acc[i].z = fmaf(xs_, z.z, acc[i].z);
                acc[i].w = fmaf(xs_, z.w, acc[i].w);
              }
            }
          }
        }
      };
      {
        // level 1: 128 threads, product pr in {0, 1} -> blocks (2pr+1, 2pr); row rp x columns c4..c4+3
        const int pr = stid >> 6, rp = (stid >> 2) & 15, c4 = (stid & 3) * 4;
        const int bi = 2 * pr + 1, bj = 2 * pr;
        float* yb = tm + 32 + pr * 16;  // Y = A_ij T_jj [16][16] in T's upper-right quarter (free)
        if (stid < 128) {
          float4 acc[1] = {};
          blk(acc, 1, am + (bi * 16 + rp) * LDC + bj * 16, tm + (bj * 16) * LDC + bj * 16 + c4, 16);
          *reinterpret_cast<float4*>(yb + rp * LDC + c4) = acc[0];
        }
        role_sync(3, NSV);
        if (stid < 128) {
          float4 acc[1] = {};
          blk(acc, 1, tm + (bi * 16 + rp) * LDC + bi * 16, yb + c4, 16);
          *reinterpret_cast<float4*>(tm + (bi * 16 + rp) * LDC + bj * 16 + c4) =
              make_float4(-acc[0].x, -acc[0].y, -acc[0].z, -acc[0].w);
        }
        role_sync(3, NSV);
      }
      {
        // level 2: all 256 threads, row rq x columns c4..c4+3 of the 32 x 32 blocks
        const int rq = stid >> 3, c4 = (stid & 7) * 4;
        {
          float4 acc[1] = {};
          blk(acc, 1, am + (32 + rq) * LDC, tm + c4, 32);
          *reinterpret_cast<float4*>(tm + rq * LDC + 32 + c4) = acc[0];
        }
        role_sync(3, NSV);
        {
          float4 acc[1] = {};
          blk(acc, 1, tm + (32 + rq) * LDC + 32, tm + 32 + c4, 32);
          *reinterpret_cast<float4*>(tm + (32 + rq) * LDC + c4) = make_float4(-acc[0].x, -acc[0].y, -acc[0].z, -acc[0].w);
        }
        role_sync(3, NSV);
      }
      // ---- S3: T diag(eta e^G n_k) and T diag(eta) as fp16 tiles (row t, 8 columns each) ----
      for (int e = stid; e < C * 8; e += NSV) {
        const int t = e >> 3, g = e & 7;
        const float4 a = *reinterpret_cast<const float4*>(tm + t * LDC + 8 * g);
        const float4 b = *reinterpret_cast<const float4*>(tm + t * LDC + 8 * g + 4);
        const float tv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float v1[8], v2[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int s = 8 * g + i;
          const float tt = s <= t ? tv[i] : 0.f;  // the upper-right quarter holds scratch
          v2[i] = tt * ETA[s];
          v1[i] = v2[i] * EG[s] * NK[s];
        }
        *reinterpret_cast<uint4*>(tp + sw(t, g)) =
            make_uint4(pack_h2(v1[0], v1[1]), pack_h2(v1[2], v1[3]), pack_h2(v1[4], v1[5]), pack_h2(v1[6], v1[7]));
        *reinterpret_cast<uint4*>(tpp + sw(t, g)) =
            make_uint4(pack_h2(v2[0], v2[1]), pack_h2(v2[2], v2[3]), pack_h2(v2[4], v2[5]), pack_h2(v2[6], v2[7]));
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      role_sync(3, NSV);
      // ---- S4: W^T = Y_k^T T'^T into the product columns, U~^T = Y_v^T T''^T into this
      //      slot's U columns (free: the chain finished chunk k-2) ------------------------
      if (stid == 0) {
        tc::tc_fence_after();
        constexpr uint32_t id4 = tc::idesc_fp16(128, 64, 1, 0);
        const uint64_t dyk = tc::sdesc_sw128(tc::smem_u32(yts + C * 128), 16384, 1024);
        const uint64_t dyv = tc::sdesc_sw128(tc::smem_u32(yv), 8192, 1024);
        const uint64_t dtp = tc::sdesc_sw128(tc::smem_u32(tp), 16, 1024);
        const uint64_t dtpp = tc::sdesc_sw128(tc::smem_u32(tpp), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
          const uint64_t ao = static_cast<uint64_t>(ks * (2048 / 16)), bo = static_cast<uint64_t>(ks * 2);
          tc::mma_bf16(tmem + T_M1, dyk + ao, dtp + bo, id4, ks > 0);
        }
        // Y_v of this chunk comes from the chain (a failed wait raises the abort flag: the
        // group's next wait gives up too)
        if (tc::mbar_wait(&bars[B_YV], k & 1, abort, p.wait_ns)) {
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks) {
            const uint64_t ao = static_cast<uint64_t>(ks * (2048 / 16)), bo = static_cast<uint64_t>(ks * 2);
            tc::mma_bf16(tmem + t_u(slot), dyv + ao, dtpp + bo, id4, ks > 0);
          }
          tc::mma_commit(&bars[B_MW]);
        }
      }
      // ---- S5: -W (fp16) into its tile, free once the chain's products of chunk k-1 that
      //      read it are done (lane = channel c, 32 tokens per thread) ----------------------
      if (!(ok = swait(B_MW, k & 1))) break;
      if (k >= 1 && !(ok = swait(B_MA, (k - 1) & 1))) break;
      tc::tc_fence_after();
      {
        const int ch = (warp - NCV / 32) >> 2;
        const int c = q4 * 32 + lane;
        uint32_t v32[32];
        tc::tmem_ld32(tmem + T_M1 + ch * 32 + lb, v32);
        tc::tmem_wait_ld();
        unsigned char* col = wt + (c >> 6) * 8192 + (c & 7) * 2;
        const int jc = (c & 63) >> 3;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int t = ch * 32 + e;
          *reinterpret_cast<__half*>(col + sw(t, jc)) = __float2half_rn(-__uint_as_float(v32[e]));
        }
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      role_sync(3, NSV);
      if (stid == 0) tc::mbar_arrive(&bars[B_PREP]);
      ++k;
      c0 += C;
      if (c0 >= len) {
        si = first_seg(si + 1);
        c0 = 0;
      }
    }
    // drain: own MMAs
    if (stid == 0) {
      tc::mma_commit(&bars[B_FINP]);
      tc::mbar_drain(&bars[B_FINP], 0);
    }
  } else {
    // ============================ state chain (128 threads) ============================
    const int ct = tid - NCV - NSV;
    const int v = q4 * 32 + lane;  // row of S (v index) = TMEM lane
    auto cwait = [&](int b, uint32_t par) -> bool {
      return role_and(2, NCH, tc::mbar_wait(&bars[b], par, abort, p.wait_ns));
    };
    // 32 fp32 values -> 16 words of fp16 pairs
    auto pack32 = [&](const uint32_t* a, uint32_t* hv) {
#pragma unroll
      for (int e = 0; e < 16; ++e) hv[e] = pack_h2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
    };
    // fp16 copy of S (the A operand of the next chunk's first products) and S scaled in
    // place by that chunk's decay e^{G_last} (before its state update), in one pass
    auto s16_and_scale = [&](float egl) {
#pragma unroll
      for (int cb = 0; cb < D; cb += 32) {
        uint32_t a[32], hv[16];
        tc::tmem_ld32(tmem + T_S + cb + lb, a);
        tc::tmem_wait_ld();
        pack32(a, hv);
        tc::tmem_st16(tmem + T_S16 + cb / 2 + lb, hv);
#pragma unroll
        for (int e = 0; e < 32; ++e) a[e] = __float_as_uint(__uint_as_float(a[e]) * egl);
        tc::tmem_st32(tmem + T_S + cb + lb, a);
      }
    };
    // S <- a state from global memory (row v), or zero; and its fp16 copy
    auto load_state = [&](const float* src) {
#pragma unroll
      for (int cb = 0; cb < D; cb += 32) {
        uint32_t a[32], hv[16];
        if (src) {
          const float4* s4 = reinterpret_cast<const float4*>(src + in_base + static_cast<int64_t>(v) * D + cb);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 f = s4[q];
            a[4 * q] = __float_as_uint(f.x);
            a[4 * q + 1] = __float_as_uint(f.y);
            a[4 * q + 2] = __float_as_uint(f.z);
            a[4 * q + 3] = __float_as_uint(f.w);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = 0u;
        }
        pack32(a, hv);
        tc::tmem_st32(tmem + T_S + cb + lb, a);
        tc::tmem_st16(tmem + T_S16 + cb / 2 + lb, hv);
      }
      tc::tmem_wait_st();
    };
    // Y_v of each chunk is made here, between the chain's own chunks (the conv group makes
    // Y_q and Y_k): raw v rows requested one chunk ahead, conv + SiLU into the Y_v tile once
    // the solve group's products of the previous chunk have read it (they complete before
    // that chunk's operands are signalled ready)
    int v_issued = 0;
    auto v_rows = [&](int s, int cc) {
      if (ct == 0) issue_rows(s, cc, 2, 3, B_RAWV);
      ++v_issued;
    };
    auto v_conv = [&](int s, int cc) -> bool {
      if (!cwait(B_RAWV, (v_issued - 1) & 1)) return false;
      if (cc == 0) {
        patch_history(ct, 2, 3);
        role_sync(2, NCH);
      }
      conv_stream(ct, 2, min(C, seg_len(s) - cc), yv, 8192, 0, nullptr);
      tc::fence_proxy_async_smem();
      role_sync(2, NCH);
      if (ct == 0) tc::mbar_arrive(&bars[B_YV]);
      return true;
    };
    auto next_chunk = [&](int& s, int& cc) {
      cc += C;
      if (cc >= seg_len(s)) {
        s = first_seg(s + 1);
        cc = 0;
      }
    };
    if (ct == 0) tc::prefetch_tmap(&vmap);
    if (!BRANCH) load_state(S0);
    bool ok = !p.stall || cwait(B_STALL, 0);  // FORK_TEST_STALL: runs out, nothing is issued
    bool s_is_start = !BRANCH;  // branch call: S holds S_P[j] (no question has updated it)
    int si = first_seg(seg_first), c0 = 0, k = 0;
    if (ok && si < seg_end) {
      v_rows(si, 0);
      ok = v_conv(si, 0);
      int s2 = si, c2 = 0;
      next_chunk(s2, c2);
      if (ok && s2 < seg_end) v_rows(s2, c2);
    }
    while (ok && si < seg_end) {
      const int start = seg_start(si), len = seg_len(si), pos0 = seg_pos0(si);
      const int n = min(C, len - c0);
      const int slot = k & 1;
      const float* G = gate(slot, G_G);
      const float* EG = gate(slot, G_EG);
      const float* GL = gate(slot, G_GL);
      const float* NQ = gate(slot, G_NQ);
      const float* NK = gate(slot, G_NK);
      unsigned char* yts = yt(slot);
      unsigned char* pb = pbt(slot);
      const bool more = c0 + C < len;  // another chunk of this segment follows
      const bool need_state = !BRANCH || more;
      // ---- C0: operands of chunk k ready; a question starts from its request's S_P ----
      if (!(ok = cwait(B_PREP, k & 1))) break;
      if (BRANCH && c0 == 0 && !s_is_start) {
        load_state(S0);
        s_is_start = true;
      }
      tc::tc_fence_before();
      role_sync(2, NCH);
      if (ct == 0) {
        tc::tc_fence_after();
        constexpr uint32_t ida = tc::idesc_fp16(128, 64, 0, 0);
        const uint64_t dw = tc::sdesc_sw128(tc::smem_u32(wt), 16, 1024);
        const uint64_t dq = tc::sdesc_sw128(tc::smem_u32(yts), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t ow = static_cast<uint64_t>((ks >> 2) * (8192 / 16) + (ks & 3) * 2);
          const uint64_t oq = static_cast<uint64_t>((ks >> 2) * (16384 / 16) + (ks & 3) * 2);
          tc::mma_f16_ts(tmem + t_u(slot), tmem + T_S16 + ks * 8, dw + ow, ida, 1u);  // U~^T - S W^T
          tc::mma_f16_ts(tmem + T_X, tmem + T_S16 + ks * 8, dq + oq, ida, ks > 0);    // S Y_q^T
        }
        tc::mma_commit(&bars[B_MA]);
      }
      // ---- C1: checkpoint; U^T to fp16 (plain, and scaled by Gamma_last n_k); X scaled by
      //      e^G n_q; S scaled by e^{G_last} ------------------------------------------------
      if (!(ok = cwait(B_MA, k & 1))) break;
      tc::tc_fence_after();
      if (!BRANCH && ck >= 0 && p.S_ckpt) {
        // state after r of this chunk's tokens (rare): e^{G_{r-1}} S0 + sum_{s<r}
        // e^{G_{r-1} - G_s} n_k,s u_s y_k,s^T
        const int r_ck = ck - pos0 - c0;
        if (r_ck >= 1 && r_ck <= n) {
          // S holds S0, or S0 e^{G_last} when the previous chunk already scaled it
          const float gr = G[r_ck - 1], s_fac = expf(c0 == 0 ? gr : gr - G[C - 1]);
#pragma unroll 1
          for (int cb = 0; cb < D; cb += 32) {
            uint32_t s32[32];
            tc::tmem_ld32(tmem + T_S + cb + lb, s32);
            tc::tmem_wait_ld();
            float acc[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[e] = s_fac * __uint_as_float(s32[e]);
            const unsigned char* ybox = yts + (cb >> 6) * 16384;
#pragma unroll 1
            for (int s = 0; s < r_ck; ++s) {
              const uint32_t u1 = tc::tmem_ld1(tmem + t_u(slot) + s + lb);  // u_s of row v (fp32)
              tc::tmem_wait_ld();
              const float us = __uint_as_float(u1) * expf(gr - G[s]) * NK[s];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint4 w = *reinterpret_cast<const uint4*>(ybox + sw(C + s, ((cb & 63) >> 3) + q));
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                  const uint32_t wv = word_of(w, e2);
                  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv));
                  acc[8 * q + 2 * e2] += us * f.x;
                  acc[8 * q + 2 * e2 + 1] += us * f.y;
                }
              }
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) p.S_ckpt[state_base + static_cast<int64_t>(v) * D + cb + e] = acc[e];
          }
        }
      }
      // U^T as fp16 pairs in place (columns 0-31 of the slot: s = 0..63, two per column) and
      // U^T diag(Gamma_last n_k) as fp16 pairs into the slot's scaled copy; 32 columns at a time
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t u32[32], lo[16], hi[16];
        tc::tmem_ld32(tmem + t_u(slot) + 32 * hh + lb, u32);
        tc::tmem_wait_ld();
        const float4* gl4 = reinterpret_cast<const float4*>(GL + 32 * hh);
        const float4* nk4 = reinterpret_cast<const float4*>(NK + 32 * hh);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 g = gl4[q], nk = nk4[q];
          lo[2 * q] = pack_h2(__uint_as_float(u32[4 * q]), __uint_as_float(u32[4 * q + 1]));
          lo[2 * q + 1] = pack_h2(__uint_as_float(u32[4 * q + 2]), __uint_as_float(u32[4 * q + 3]));
          hi[2 * q] = pack_h2(__uint_as_float(u32[4 * q]) * g.x * nk.x, __uint_as_float(u32[4 * q + 1]) * g.y * nk.y);
          hi[2 * q + 1] =
              pack_h2(__uint_as_float(u32[4 * q + 2]) * g.z * nk.z, __uint_as_float(u32[4 * q + 3]) * g.w * nk.w);
        }
        tc::tmem_st16(tmem + t_u(slot) + 16 * hh + lb, lo);  // the columns just read
        tc::tmem_st16(tmem + t_ug(slot) + 16 * hh + lb, hi);
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t v32[32];
        tc::tmem_ld32(tmem + T_X + q * 32 + lb, v32);
        tc::tmem_wait_ld();
        const float4* eg4 = reinterpret_cast<const float4*>(EG + q * 32);
        const float4* nq4 = reinterpret_cast<const float4*>(NQ + q * 32);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 g = eg4[e4], nq = nq4[e4];
          v32[4 * e4] = __float_as_uint(__uint_as_float(v32[4 * e4]) * g.x * nq.x);
          v32[4 * e4 + 1] = __float_as_uint(__uint_as_float(v32[4 * e4 + 1]) * g.y * nq.y);
          v32[4 * e4 + 2] = __float_as_uint(__uint_as_float(v32[4 * e4 + 2]) * g.z * nq.z);
          v32[4 * e4 + 3] = __float_as_uint(__uint_as_float(v32[4 * e4 + 3]) * g.w * nq.w);
        }
        tc::tmem_st32(tmem + T_X + q * 32 + lb, v32);
      }
      if (need_state && c0 == 0) {  // later chunks of the segment: scaled at the end of the one before
        const float egl = EG[C - 1];
#pragma unroll
        for (int cb = 0; cb < D; cb += 32) {
          uint32_t v32[32];
          tc::tmem_ld32(tmem + T_S + cb + lb, v32);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v32[e] = __float_as_uint(__uint_as_float(v32[e]) * egl);
          tc::tmem_st32(tmem + T_S + cb + lb, v32);
        }
        s_is_start = false;
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      role_sync(2, NCH);
      // ---- C2: O^T += U^T P^T and S += (U^T diag(Gamma_last n_k)) Y_k --------------------
      if (ct == 0) {
        tc::tc_fence_after();
        constexpr uint32_t id5 = tc::idesc_fp16(128, 64, 0, 0);
        constexpr uint32_t id6 = tc::idesc_fp16(128, 128, 0, 1);
        const uint64_t dp = tc::sdesc_sw128(tc::smem_u32(pb), 16, 1024);
        const uint64_t dk = tc::sdesc_sw128(tc::smem_u32(yts + C * 128), 16384, 1024);
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks)
          tc::mma_f16_ts(tmem + T_X, tmem + t_u(slot) + ks * 8, dp + static_cast<uint64_t>(ks * 2), id5, 1u);
        if (need_state)
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks)
            tc::mma_f16_ts(tmem + T_S, tmem + t_ug(slot) + ks * 8, dk + static_cast<uint64_t>(ks * (2048 / 16)),
                           id6, 1u);
        tc::mma_commit(&bars[B_MB]);
      }
      // ---- C3: output rows, staged 32 tokens at a time in this slot's P tile (read by the
      //      products just completed).  Thread v holds column v; lane pairs swap values so
      //      that each shared-memory store carries two neighbouring columns of one token; odd
      //      rows are rotated by 64 bytes so the two tokens of one store use different banks.
      if (!(ok = cwait(B_MB, k & 1))) break;
      tc::tc_fence_after();
      // the products of this chunk are done: its row tiles, gates and U slot are free
      tc::mbar_arrive(&bars[B_EPI0 + slot]);
      {
        const bool odd = lane & 1;
        const int v0 = v & ~1;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t v32[32];
          tc::tmem_ld32(tmem + T_X + q * 32 + lb, v32);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            // even lane: (token t, columns v, v+1); odd lane: (token t+1, columns v-1, v)
            const float mine_t = __uint_as_float(v32[e]), mine_t1 = __uint_as_float(v32[e + 1]);
            const float other = __shfl_xor_sync(0xffffffffu, odd ? mine_t : mine_t1, 1);
            const int t = e + (odd ? 1 : 0);
            const __nv_bfloat162 pr =
                odd ? __floats2bfloat162_rn(other, mine_t1) : __floats2bfloat162_rn(mine_t, other);
            *reinterpret_cast<__nv_bfloat162*>(pb + t * (D * 2) + ((v0 * 2 + (t & 1) * 64) & (D * 2 - 1))) = pr;
          }
          role_sync(2, NCH);
          const int cq = ct & 15;  // 16-byte piece of a 256-byte row
#pragma unroll
          for (int pass = 0; pass < 4; ++pass) {
            const int t = pass * 8 + (ct >> 4);
            if (q * 32 + t < n) {
              const uint4 val =
                  *reinterpret_cast<const uint4*>(pb + t * (D * 2) + ((cq * 16 + (t & 1) * 64) & (D * 2 - 1)));
              *reinterpret_cast<uint4*>(p.o + (static_cast<int64_t>(start + c0 + q * 32 + t) * H + h) * D + cq * 8) =
                  val;
            }
          }
          role_sync(2, NCH);
        }
      }
      if (more) {  // the next chunk of this segment: its decay is known once its gates are
        if (!(ok = cwait(B_GATE, (k + 1) & 1))) break;
        s16_and_scale(gate(slot ^ 1, G_EG)[C - 1]);
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      tc::mbar_arrive(&bars[B_PF0 + slot]);  // the P tile (output staging) is free
      ++k;
      next_chunk(si, c0);
      // Y_v of the next chunk; then the raw v rows of the one after it
      if (si < seg_end) {
        if (!(ok = v_conv(si, c0))) break;
        int s2 = si, c2 = c0;
        next_chunk(s2, c2);
        if (s2 < seg_end) v_rows(s2, c2);
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
      // raw v rows still in flight after an abort (the last ones issued)
      if (!ok && v_issued > 0) tc::mbar_drain(&bars[B_RAWV], (v_issued - 1) & 1);
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
      return hist[((static_cast<int64_t>(in_idx * (KW - 1) + r) * 3 + s) * H + h) * D + c];
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
  // boxes of 64 channels x 1 head x HR rows, 128-byte swizzle (zero fill outside the tensor)
  for (int i = 0; i < 3; ++i)
    if (!encode_map_3d(&maps[i], src[i], D, p.H, p.L.T_cap, 64, 1, HR, true)) return FORK_ECUDA;
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
