// Fork-masked varlen attention on the 5th-generation tensor cores (tcgen05).
//
// Visibility (rainbus summary "方法步骤详情" step 2; onedev "무엇과 다른가"):
// key y is visible to query x iff j_y = j_x, c_y in {0, c_x}, t_y <= t_x and,
// for a sliding-window layer, t_x - t_y < W.  A query tile (128 rows =
// tile_tokens tokens x the Hq/Hkv heads that share one kv head) reads at most
// three contiguous key ranges: the request's prefix rows kept outside the
// stream, its trunk segment, and for a question its own branch.  Inside a
// range, key u (position p0 + u) is visible to query position t iff u < len,
// p0 + u <= t and (W == 0 or t - p0 - u < W).  Key tiles are aligned to the
// range start and query tiles to the segment start: every output element is
// produced by the same sequence of operations whatever else the round holds.
//
// One CTA = one query tile x one kv head, 6 warps:
//   warp 4 (one lane)  TMA producer: Q once, then K/V tiles into a 2-stage ring;
//   warp 5 (one lane)  MMA issuer: S = Q K^T into one of two TMEM buffers,
//                      O += P V into a TMEM accumulator; TMEM owner;
//   warps 0-3          one query row per thread: S from TMEM, mask, online
//                      softmax in the log2 domain (the running maximum is only
//                      moved when it grows by more than 2^8, so O is rescaled
//                      rarely), P (bf16) into shared memory, final O / l.
// Operands are bf16 in 128-byte-swizzled shared memory, accumulation f32 in
// TMEM.  Every wait is bounded; on a timeout the CTA raises the status bit,
// drains its own copies and MMAs, frees TMEM and exits.
#include "fork_attn.cuh"
#include "tc_ptx.cuh"

namespace fork {

namespace {

constexpr int kRows = 128;   // query rows per CTA
constexpr int kKeys = 128;   // keys per tile
constexpr int kBox = 128 * 128;  // bytes of one 128-row x 64-element bf16 box
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescale = 8.f;  // move the running max only when it grows by > 2^8

template <int D>
struct TcLayout {
  static constexpr int NB = D / 64;  // 64-element boxes per row
  static constexpr int Q = 0;
  static constexpr int K = Q + NB * kBox;           // 2 stages
  static constexpr int V = K + 2 * NB * kBox;       // 2 stages
  static constexpr int P = V + 2 * NB * kBox;       // 2 boxes (128 keys)
  static constexpr int BAR = P + 2 * kBox;
  static constexpr int BYTES = BAR + 256;
  static constexpr int SMEM = (BYTES + 1024 > 120 * 1024 ? BYTES + 1024 : 120 * 1024);  // one CTA per SM
};

enum Bar { B_QFULL = 0, B_KFULL0, B_KFULL1, B_VFULL0, B_VFULL1, B_KEMPTY0, B_KEMPTY1, B_VEMPTY0,
           B_VEMPTY1, B_SFULL0, B_SFULL1, B_SFREE0, B_SFREE1, B_PFULL, B_ODONE, B_FIN, B_COUNT };

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x on the SFU (flush-to-zero; 2^-inf = 0)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// byte offset of element e (0 <= e < D) of row r inside a [128 x D] K-major
// SW128 tile made of D/64 boxes
__device__ __forceinline__ int sw128_off(int r, int e) {
  const int b = e >> 6, ce = e & 63;
  return b * kBox + r * 128 + ((((ce >> 3) ^ (r & 7))) << 4) + ((ce & 7) << 1);
}

}  // namespace

struct TcParams {
  const int32_t* meta;
  MetaLayout L;
  uint16_t* o;
  int Hq, Hkv, G, prefix_rows, window;
  float scale_log2;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap pkmap,
                   const __grid_constant__ CUtensorMap pvmap, const TcParams p) {
  using LY = TcLayout<D>;
  constexpr int NB = LY::NB;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int32_t* meta = p.meta;
  const MetaLayout& L = p.L;
  if (meta[H_VALID] == 0) return;
  const int w = blockIdx.x;
  if (w >= meta[H_NWORK]) return;
  const int g = blockIdx.y;
  const int G = p.G;
  const int tile = kRows / G;
  const int s = meta[L.work_seg + w];
  const int off = meta[L.work_off + w];
  const int seg_start = meta[L.seg_start + s];
  const int seg_len = meta[L.seg_len + s];
  const int seg_pos0 = meta[L.seg_pos0 + s];
  const int j = meta[L.seg_req + s];
  const int c = meta[L.seg_branch + s];
  const int n = min(tile, seg_len - off);
  const int tx_min = seg_pos0 + off;
  const int tx_max = seg_pos0 + off + n - 1;

  // ---- key ranges in fixed slots: 0 prefix rows, 1 trunk, 2 own branch --------------
  // (an absent range has length 0; fixed slots keep every range variable in registers)
  const int pl = meta[L.req_prefix_len + j];
  const int poff = pl > 0 ? meta[L.req_prefix_off + j] : 0;
  if (pl > 0 && poff + pl > p.prefix_rows) {
    if (threadIdx.x == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_BAD_PREFIX);
    return;
  }
  const int r_row0_0 = poff, r_len_0 = pl, r_pos0_0 = 0;
  const int r_row0_1 = meta[L.seg_trunk_start + s], r_len_1 = meta[L.seg_trunk_len + s], r_pos0_1 = pl;
  const int r_row0_2 = seg_start, r_len_2 = c > 0 ? seg_len : 0, r_pos0_2 = seg_pos0;
  auto tiles = [&](int len, int pos0, int& lo_t, int& cnt_t) {
    lo_t = 0;
    cnt_t = 0;
    if (len <= 0) return;
    const int umax = min(len - 1, tx_max - pos0);
    const int umin = p.window > 0 ? max(0, tx_min - p.window + 1 - pos0) : 0;
    if (umax >= umin) {
      lo_t = umin / kKeys;
      cnt_t = umax / kKeys - lo_t + 1;
    }
  };
  int lo0, cnt0, lo1, cnt1, lo2, cnt2;
  tiles(r_len_0, r_pos0_0, lo0, cnt0);
  tiles(r_len_1, r_pos0_1, lo1, cnt1);
  tiles(r_len_2, r_pos0_2, lo2, cnt2);
  const int total = cnt0 + cnt1 + cnt2;
  if (total == 0) return;  // cannot happen for a valid tile (a token sees itself)
  // flat key-tile index f -> range slot r, first key row, length, first position, tile t
  struct KT {
    int r, row0, len, pos0, t;
  };
  auto key_tile = [&](int f) -> KT {
    if (f < cnt0) return {0, r_row0_0, r_len_0, r_pos0_0, lo0 + f};
    f -= cnt0;
    if (f < cnt1) return {1, r_row0_1, r_len_1, r_pos0_1, lo1 + f};
    f -= cnt1;
    return {2, r_row0_2, r_len_2, r_pos0_2, lo2 + f};
  };

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::BAR + B_COUNT * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + LY::BAR + B_COUNT * 8 + 8);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    tc::mbar_init(&bars[B_QFULL], 1);
    for (int k = 0; k < 2; ++k) {
      tc::mbar_init(&bars[B_KFULL0 + k], 1);
      tc::mbar_init(&bars[B_VFULL0 + k], 1);
      tc::mbar_init(&bars[B_KEMPTY0 + k], 1);
      tc::mbar_init(&bars[B_VEMPTY0 + k], 1);
    }
    tc::mbar_init(&bars[B_SFULL0], 1);
    tc::mbar_init(&bars[B_SFULL1], 1);
    tc::mbar_init(&bars[B_SFREE0], 128);
    tc::mbar_init(&bars[B_SFREE1], 128);
    tc::mbar_init(&bars[B_PFULL], 128);
    tc::mbar_init(&bars[B_ODONE], 1);
    tc::mbar_init(&bars[B_FIN], 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto tm_s = [&](int st) -> uint32_t { return tmem + static_cast<uint32_t>(st) * 128u; };
  const uint32_t tm_o = tmem + 256;
  unsigned char* sQ = smem + LY::Q;
  unsigned char* sK = smem + LY::K;
  unsigned char* sV = smem + LY::V;
  unsigned char* sP = smem + LY::P;

  if (warp == 4) {
    // ===================== TMA producer =====================
    if (lane == 0) {
      tc::prefetch_tmap(&qmap);
      tc::prefetch_tmap(&kmap);
      tc::prefetch_tmap(&vmap);
      if (pl > 0) {
        tc::prefetch_tmap(&pkmap);
        tc::prefetch_tmap(&pvmap);
      }
      tc::mbar_expect_tx(&bars[B_QFULL], NB * kBox);
      for (int b = 0; b < NB; ++b) tc::tma_load_3d(sQ + b * kBox, &qmap, &bars[B_QFULL], b * 64, g * G, seg_start + off);
      // K_f waits for QK_{f-2} (its slot's previous reader), V_f for PV_{f-2}
      int issued = 0;
      for (int f = 0; f < total; ++f) {
        const int st = f & 1;
        const KT kt = key_tile(f);
        const CUtensorMap* km = kt.r == 0 ? &pkmap : &kmap;
        const CUtensorMap* vm = kt.r == 0 ? &pvmap : &vmap;
        const int row = kt.row0 + kt.t * kKeys;
        if (f >= 2 && !tc::mbar_wait(&bars[B_KEMPTY0 + st], ((f >> 1) - 1) & 1, abort)) break;
        tc::mbar_expect_tx(&bars[B_KFULL0 + st], NB * kBox);
        for (int b = 0; b < NB; ++b) tc::tma_load_3d(sK + (st * NB + b) * kBox, km, &bars[B_KFULL0 + st], b * 64, g, row);
        if (f >= 2 && !tc::mbar_wait(&bars[B_VEMPTY0 + st], ((f >> 1) - 1) & 1, abort)) break;
        tc::mbar_expect_tx(&bars[B_VFULL0 + st], NB * kBox);
        for (int b = 0; b < NB; ++b) tc::tma_load_3d(sV + (st * NB + b) * kBox, vm, &bars[B_VFULL0 + st], b * 64, g, row);
        issued = f + 1;
      }
      // drain: the last loads issued complete by themselves
      tc::mbar_wait(&bars[B_QFULL], 0, abort);
      for (int f = max(0, issued - 2); f < issued; ++f) {
        tc::mbar_wait(&bars[B_KFULL0 + (f & 1)], (f >> 1) & 1, abort);
        tc::mbar_wait(&bars[B_VFULL0 + (f & 1)], (f >> 1) & 1, abort);
      }
    }
  } else if (warp == 5) {
    // ===================== MMA issuer =====================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16(128, kKeys, 0, 0);
      constexpr uint32_t idesc_pv = tc::idesc_bf16(128, D, 0, 1);
      // descriptors are built once; the start-address field (16-byte units) is then
      // advanced by constants: +2 per 32-byte k step, +kBox/16 per box
      const uint64_t dq = tc::sdesc_sw128(tc::smem_u32(sQ), 16, 1024);
      const uint64_t dk = tc::sdesc_sw128(tc::smem_u32(sK), 16, 1024);
      const uint64_t dp = tc::sdesc_sw128(tc::smem_u32(sP), 16, 1024);
      const uint64_t dv = tc::sdesc_sw128(tc::smem_u32(sV), kBox, 1024);
      constexpr uint64_t kBoxU = kBox / 16, kStageU = NB * kBox / 16;
      bool ok = tc::mbar_wait(&bars[B_QFULL], 0, abort);
      auto issue_pv = [&](int f) -> bool {
        const int st = f & 1;
        if (!tc::mbar_wait(&bars[B_VFULL0 + st], (f >> 1) & 1, abort)) return false;
        if (!tc::mbar_wait(&bars[B_PFULL], f & 1, abort)) return false;
        tc::tc_fence_after();
#pragma unroll
        for (int step = 0; step < kKeys / 16; ++step)
          tc::mma_bf16(tm_o, dp + (step >> 2) * kBoxU + (step & 3) * 2, dv + st * kStageU + step * (2048 / 16),
                       idesc_pv, (f > 0 || step > 0) ? 1u : 0u);
        tc::mma_commit(&bars[B_ODONE]);
        tc::mma_commit(&bars[B_VEMPTY0 + st]);
        return true;
      };
      for (int f = 0; ok && f < total; ++f) {
        const int st = f & 1;
        if (!tc::mbar_wait(&bars[B_KFULL0 + st], (f >> 1) & 1, abort)) { ok = false; break; }
        if (f >= 2 && !tc::mbar_wait(&bars[B_SFREE0 + st], ((f >> 1) - 1) & 1, abort)) { ok = false; break; }
        tc::tc_fence_after();
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_bf16(tm_s(st), dq + b * kBoxU + k * 2, dk + st * kStageU + b * kBoxU + k * 2, idesc_qk,
                         (b | k) ? 1u : 0u);
        tc::mma_commit(&bars[B_SFULL0 + st]);
        tc::mma_commit(&bars[B_KEMPTY0 + st]);
        if (f >= 1 && !issue_pv(f - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(total - 1);
      // every MMA issued by this thread has completed before TMEM is released
      tc::mma_commit(&bars[B_FIN]);
      tc::mbar_wait(&bars[B_FIN], 0, abort);
    }
  } else {
    // ===================== softmax warps (row = tid) =====================
    const int row = tid;
    const int tok = row / G, hl = row % G;
    const int tx = tx_min + tok;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    bool ok = true;
    float m_used = -INFINITY, l = 0.f;
    const float sl2 = p.scale_log2;
    for (int f = 0; ok && f < total; ++f) {
      const int st = f & 1;
      ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_SFULL0 + st], (f >> 1) & 1, abort));
      if (!ok) break;
      tc::tc_fence_after();
      float sv[kKeys];
      {
        uint32_t rawv[kKeys];
#pragma unroll
        for (int i = 0; i < kKeys / 32; ++i) tc::tmem_ld32(tm_s(st) + lane_base + i * 32, rawv + i * 32);
        tc::tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < kKeys; ++cc) sv[cc] = __uint_as_float(rawv[cc]);
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&bars[B_SFREE0 + st]);
      const KT kt = key_tile(f);
      const int u0 = kt.t * kKeys;
      const int len = kt.len, p0 = kt.pos0;
      const bool need_mask = (u0 + kKeys > len) || (p0 + u0 + kKeys - 1 > tx_min) ||
                             (p.window > 0 && tx_max - (p0 + u0) >= p.window);
      if (need_mask) {
        // key u0+cc visible iff inside the range, not after the query, inside the window
        const int lim_len = len - u0;          // cc < lim_len
        const int lim_causal = tx - p0 - u0;   // cc <= lim_causal
        const int lim_win = p.window > 0 ? tx - p0 - u0 - p.window : -0x40000000;  // cc > lim_win
#pragma unroll
        for (int cc = 0; cc < kKeys; ++cc)
          if (cc >= lim_len || cc > lim_causal || cc <= lim_win) sv[cc] = -INFINITY;
      }
      // row maximum (raw scores; the scale is positive)
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = sv[e];
#pragma unroll
      for (int cc = 8; cc < kKeys; ++cc) mx[cc & 7] = fmaxf(mx[cc & 7], sv[cc]);
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
      const bool resc = mt > m_used + kRescale;
      const float m_new = resc ? mt : m_used;
      const float base = (m_new == -INFINITY) ? 0.f : m_new;
      const float factor = resc ? exp2f(m_used - base) : 1.f;  // 0 when nothing was accumulated
      // p = 2^(s*scale*log2e - base), summed with independent partial sums
      float ps[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) ps[e] = 0.f;
#pragma unroll
      for (int cc = 0; cc < kKeys; ++cc) {
        sv[cc] = fast_exp2(fmaf(sv[cc], sl2, -base));
        ps[cc & 7] += sv[cc];
      }
      const float rs = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      l = l * factor + rs;
      m_used = m_new;
      if (f >= 1) {
        ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_ODONE], (f - 1) & 1, abort));
        if (!ok) break;
        tc::tc_fence_after();
        if (__any_sync(0xffffffffu, factor != 1.f)) {
#pragma unroll
          for (int i = 0; i < D / 32; ++i) {
            uint32_t ov[32];
            tc::tmem_ld32(tm_o + lane_base + i * 32, ov);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * factor);
            tc::tmem_st32(tm_o + lane_base + i * 32, ov);
          }
          tc::tmem_wait_st();
        }
      }
      // key rows past the range end may be pad rows of the stream: zero them in V
      if (u0 + kKeys > len) {
        ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_VFULL0 + st], (f >> 1) & 1, abort));
        if (!ok) break;
        const int valid_rows = max(0, len - u0);
        if (row >= valid_rows) {
          unsigned char* vrow = sV + st * NB * kBox + row * 128;
#pragma unroll
          for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(vrow + b * kBox + q * 16) = make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int q = 0; q < kKeys / 8; ++q) {
        uint4 v4;
        v4.x = pack_bf16(sv[q * 8 + 0], sv[q * 8 + 1]);
        v4.y = pack_bf16(sv[q * 8 + 2], sv[q * 8 + 3]);
        v4.z = pack_bf16(sv[q * 8 + 4], sv[q * 8 + 5]);
        v4.w = pack_bf16(sv[q * 8 + 6], sv[q * 8 + 7]);
        *reinterpret_cast<uint4*>(sP + sw128_off(row, q * 8)) = v4;
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(&bars[B_PFULL]);
    }
    if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_ODONE], (total - 1) & 1, abort));
    if (ok) {
      tc::tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* orow = p.o + (static_cast<int64_t>(seg_start + off + tok) * p.Hq + g * G + hl) * D;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        uint32_t ov[32];
        tc::tmem_ld32(tm_o + lane_base + i * 32, ov);
        tc::tmem_wait_ld();
        if (tok < n) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v4;
            v4.x = pack_bf16(__uint_as_float(ov[q * 8 + 0]) * inv, __uint_as_float(ov[q * 8 + 1]) * inv);
            v4.y = pack_bf16(__uint_as_float(ov[q * 8 + 2]) * inv, __uint_as_float(ov[q * 8 + 3]) * inv);
            v4.z = pack_bf16(__uint_as_float(ov[q * 8 + 4]) * inv, __uint_as_float(ov[q * 8 + 5]) * inv);
            v4.w = pack_bf16(__uint_as_float(ov[q * 8 + 6]) * inv, __uint_as_float(ov[q * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + i * 32 + q * 8) = v4;
          }
        }
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (*abort && tid == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_TIMEOUT);
  if (warp == 5) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- host side -------------------------------------------------------------------

template <int D>
int launch_attn_tc(const AttnParams& a, const CUtensorMap* maps, int grid_x, cudaStream_t s) {
  using LY = TcLayout<D>;
  if (cuda_rc(cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM)) != FORK_OK)
    return FORK_ECUDA;
  TcParams p;
  p.meta = a.meta;
  p.L = a.L;
  p.o = a.o;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.G;
  p.prefix_rows = a.prefix_rows;
  p.window = a.window;
  p.scale_log2 = a.scale_log2;
  dim3 grid(grid_x, a.Hkv);
  attn_tc_kernel<D><<<grid, kThreads, LY::SMEM, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  return cuda_rc(cudaGetLastError());
}

template int launch_attn_tc<64>(const AttnParams&, const CUtensorMap*, int, cudaStream_t);
template int launch_attn_tc<128>(const AttnParams&, const CUtensorMap*, int, cudaStream_t);

}  // namespace fork
