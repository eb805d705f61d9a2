// Fork-masked varlen attention on the 5th-generation tensor cores (tcgen05).
//
// Visibility (rainbus summary "方法步骤详情" step 2; onedev "무엇과 다른가"):
// key y is visible to query x iff j_y = j_x, c_y in {0, c_x}, t_y <= t_x and,
// for a sliding-window layer, t_x - t_y < W.  The queries of one work item
// (tile_tokens tokens of one segment x the Hq/Hkv heads that share a kv head)
// read at most three contiguous key ranges: the request's prefix rows kept
// outside the stream, its trunk segment, and for a question its own branch.
// Inside a range, key u (position p0 + u) is visible to query position t iff
// u < len, p0 + u <= t and (W == 0 or t - p0 - u < W).  Key tiles are aligned
// to the range start and query tiles to the segment start: every output
// element is produced by the same sequence of operations whatever else the
// round holds.
// Token forests (rainbus "未来方向" (2): a draft-token tree runs in the same flat
// stream as the request tree): the segments are the nodes, and a node's queries
// read the rows of each of its ancestors (root first) and then its own, all in
// place in the stream; positions continue along the path, so the same per-range
// rule applies (kernel instance with kForestRanges range slots).
//
// A work item x one kv head = up to two 128-row query tiles (rows = token x
// grouped head) that share every K/V tile.  The kernel is persistent: one CTA
// per SM takes items longest first (blockIdx.x, then the next unclaimed one
// through an atomic counter), 10 warps:
//   warp 1 (one lane)   claims items and hands them to the other warps through
//                       a ring in shared memory; TMA producer: both Q tiles of
//                       an item (once the previous item's QK^T products have
//                       read theirs), then K and V tiles into two 2-stage rings
//                       (K and V of a slot complete one barrier; slots are freed
//                       by their readers), running on into the next item;
//   warp 0              MMA issuer (lane 0) and TMEM owner.  Per key tile j:
//                       O_0 += P_0(j-1) V(j-1), S_0 = Q_0 K(j)^T, then the same
//                       for tile 1, so one tile's softmax overlaps the other
//                       tile's products; an item's first PV products overwrite
//                       O_t once the previous item's rows have been read;
//   warps 2-5 / 6-9     rotary embedding of tile 0 / 1 in shared memory, then
//                       its softmax, one query row per thread (warp w reads
//                       TMEM lanes 32 (w mod 4) ..; row = tid mod 128): S from
//                       TMEM, mask, online softmax in the log2 domain (the
//                       running maximum only moves when it grows by more than
//                       2^8, so O is rescaled rarely), P as fp16 written back
//                       into the TMEM columns of S, where the PV product reads
//                       it as its A operand; at the end O / l.  The next item's
//                       query tiles are rotated before this item's output rows
//                       are written.
// TMEM: S/P of tile t at columns 128t, O_t at 256 + t*D (512 columns).
// QK^T operands are bf16, PV operands fp16 (values converted once per call),
// accumulation f32 in TMEM.  Every wait is bounded; on a timeout the CTA raises
// the status bit, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda_fp16.h>

#include "fork_attn.cuh"
#include "tc_ptx.cuh"

namespace fork {

namespace {

constexpr int kRows = 128;   // query rows per MMA tile
constexpr int kKeys = 128;   // keys per tile
constexpr int kBox = 128 * 128;  // bytes of one 128-row x 64-element bf16 box
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescale = 8.f;  // move the running max only when it grows by > 2^8
constexpr int kVStages = 2;      // V ring depth = K ring depth (a third slot measured no faster)
static_assert(kVStages == 2, "K and V tiles share the slot barriers");

template <int D>
struct TcLayout {
  static constexpr int NB = D / 64;  // 64-element boxes per row
  static constexpr int Q = 0;                        // 2 query tiles
  static constexpr int K = Q + 2 * NB * kBox;        // 2 stages
  static constexpr int V = K + 2 * NB * kBox;        // 2 stages
  static constexpr int BAR = V + kVStages * NB * kBox;  // barriers, TMEM address, abort flag, tables
  static constexpr int BYTES = BAR + 2048;
  static constexpr int SMEM = (BYTES + 1024 > 120 * 1024 ? BYTES + 1024 : 120 * 1024);  // one CTA per SM
};

// B_KVFULLs: K and V tile f both landed in slot s = f mod 2 (one wait for the issuer)
enum Bar { B_QFULL = 0, B_QEMPTY, B_KVFULL0, B_KVFULL1, B_KEMPTY0, B_KEMPTY1, B_VEMPTY0, B_VEMPTY1, B_SFULL0,
           B_SFULL1, B_PFULL0, B_PFULL1, B_OFULL0, B_OFULL1, B_OFREE0, B_OFREE1, B_FIN, B_QROT, B_STALL,
           B_ITEMF0, B_ITEMF1, B_ITEMF2, B_ITEMF3, B_ITEME0, B_ITEME1, B_ITEME2, B_ITEME3, B_COUNT };
constexpr int kItemRing = 4;  // claimed work items handed from the producer to the other roles
constexpr int kRoundRanges = 3;                           // prefix, trunk, own branch
constexpr int kForestRanges = FORK_FOREST_MAX_DEPTH + 1;  // ancestors root first, then the node

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^a, 2^b of two scores on the SFU in one half-precision pair operation (2^-inf = 0),
// returned as an fp16 pair (lower half = a): the P operand of the PV product, whose
// values are fp16 too.  The arguments are at most 8 (the running maximum lags by at most
// that), so the results stay below 256.
__device__ __forceinline__ uint32_t exp2_pair(float a, float b) {
  const __half2 x = __floats2half2_rn(a, b);
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(*reinterpret_cast<const uint32_t*>(&x)));
  return y;
}
__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// max(a, b, c) in one instruction
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// tcgen05.mma kind::f16 with A (bf16, 2 per 32-bit column) read from TMEM
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

}  // namespace

struct TcParams {
  const int32_t* meta;
  MetaLayout L;
  uint16_t* o;
  const float2* rope_hi;  // (cos, sin) tables of the rotary embedding (rotate_q)
  const float2* rope_lo;
  int Hq, Hkv, G, prefix_rows, window, two_tiles, rotate_q, rope_hi_rows, checks, stall;
  float scale_log2;
  uint64_t wait_ns;
  int* work_ctr;  // work items claimed after the first gridDim.x (zeroed before the launch)
};

// Rotary embedding of one query row held in a 128-byte-swizzled tile (boxes of 64
// elements, 128 bytes per row): pairs (i, i + D/2) at position tpos, 8 pairs per step
// (one 16-byte piece of each half; both pieces sit at the same swizzled chunk when D =
// 128).  (cos, sin) by angle addition from the two-level table, as in the rotation pass.
template <int D>
__device__ __forceinline__ void rotate_q_row(unsigned char* tile, int row, int tpos, const float2* __restrict__ hi,
                                             const float2* __restrict__ lo) {
  constexpr int HALF = D / 2;
  const float4* A = reinterpret_cast<const float4*>(hi + static_cast<int64_t>(tpos >> 6) * HALF);
  const float4* B = reinterpret_cast<const float4*>(lo + static_cast<int64_t>(tpos & 63) * HALF);
#pragma unroll
  for (int c = 0; c < HALF / 8; ++c) {
    const int ea = 8 * c, eb = ea + HALF;
    uint4* pa = reinterpret_cast<uint4*>(tile + (ea >> 6) * kBox + row * 128 + ((((ea & 63) >> 3) ^ (row & 7)) << 4));
    uint4* pb = reinterpret_cast<uint4*>(tile + (eb >> 6) * kBox + row * 128 + ((((eb & 63) >> 3) ^ (row & 7)) << 4));
    const uint4 xa = *pa, xb = *pb;
    const uint32_t aw[4] = {xa.x, xa.y, xa.z, xa.w}, bw[4] = {xb.x, xb.y, xb.z, xb.w};
    uint32_t oa[4], ob[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // pairs ea+2q, ea+2q+1
      const float4 a4 = A[c * 4 + q], b4 = B[c * 4 + q];
      float ya[2], yb[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float ac = e ? a4.z : a4.x, as = e ? a4.w : a4.y;
        const float bc = e ? b4.z : b4.x, bs = e ? b4.w : b4.y;
        const float cs = ac * bc - as * bs, sn = as * bc + ac * bs;
        const float x0 = bf2f(static_cast<uint16_t>(e ? aw[q] >> 16 : aw[q] & 0xffffu));
        const float x1 = bf2f(static_cast<uint16_t>(e ? bw[q] >> 16 : bw[q] & 0xffffu));
        ya[e] = x0 * cs - x1 * sn;
        yb[e] = x1 * cs + x0 * sn;
      }
      oa[q] = static_cast<uint32_t>(f2bf(ya[0])) | (static_cast<uint32_t>(f2bf(ya[1])) << 16);
      ob[q] = static_cast<uint32_t>(f2bf(yb[0])) | (static_cast<uint32_t>(f2bf(yb[1])) << 16);
    }
    *pa = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    *pb = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  }
}

// One work item of a call: kv head g x entry r of the longest-first order (q = g n_work + r).  Its query
// tokens, and its key ranges in fixed slots (an absent range has length 0): for a round
// (NR = kRoundRanges) 0 prefix rows kept outside the stream, 1 trunk, 2 own branch; for a
// forest (NR = kForestRanges) the node's ancestors, root first, then the node itself.  The
// producer computes it from the tables and hands it to the other roles.
template <int NR>
struct AttnItem {
  int ok, status;  // status: the bit to raise when the item is skipped (ok == 0)
  int g, seg_start, off, n_all, ntiles, tx_min, total;
  int row0[NR], len[NR], pos0[NR], lo[NR], cnt[NR];
};

// first key tile and tile count of every range slot: the keys of the range at positions
// in [tx_min - W + 1, tx_max] (no lower bound without a window), in tiles aligned to the
// range start
template <int NR>
__device__ __forceinline__ void item_key_tiles(AttnItem<NR>& it, int tx_max, int window) {
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    it.lo[k] = 0;
    it.cnt[k] = 0;
    if (it.len[k] > 0) {
      const int umax = min(it.len[k] - 1, tx_max - it.pos0[k]);
      const int umin = window > 0 ? max(0, it.tx_min - window + 1 - it.pos0[k]) : 0;
      if (umax >= umin) {
        it.lo[k] = umin / kKeys;
        it.cnt[k] = umax / kKeys - it.lo[k] + 1;
      }
    }
    it.total += it.cnt[k];
  }
}

__device__ __forceinline__ AttnItem<kRoundRanges> attn_item(const int32_t* meta, const MetaLayout& L,
                                                            const TcParams& p, int q) {
  AttnItem<kRoundRanges> it;
  // head-major: the CTAs running at one time mostly share a kv head, so the K/V tiles
  // they re-read stay in L2
  const int nw = meta[H_NWORK];
  it.g = q / nw;
  const int r = q - it.g * nw;
  it.ok = 0;
  it.status = 0;
  it.total = 0;
  const int w = meta[L.work_order + r];
  if (p.checks && !attn_item_in_bounds(meta, L, w)) {
    it.status = FORK_STATUS_CHECK;
    return it;
  }
  const int s = meta[L.work_seg + w];
  it.off = meta[L.work_off + w];
  it.seg_start = meta[L.seg_start + s];
  const int seg_len = meta[L.seg_len + s];
  const int seg_pos0 = meta[L.seg_pos0 + s];
  const int j = meta[L.seg_req + s];
  const int c = meta[L.seg_branch + s];
  const int tile = kRows / p.G;
  it.n_all = min(p.two_tiles ? 2 * tile : tile, seg_len - it.off);
  it.ntiles = it.n_all > tile ? 2 : 1;
  it.tx_min = seg_pos0 + it.off;
  const int tx_max = it.tx_min + it.n_all - 1;
  const int pl = meta[L.req_prefix_len + j];
  const int poff = pl > 0 ? meta[L.req_prefix_off + j] : 0;
  if (pl > 0 && poff + pl > p.prefix_rows) {
    it.status = FORK_STATUS_BAD_PREFIX;
    return it;
  }
  it.row0[0] = poff;
  it.len[0] = pl;
  it.pos0[0] = 0;
  it.row0[1] = meta[L.seg_trunk_start + s];
  it.len[1] = meta[L.seg_trunk_len + s];
  it.pos0[1] = pl;
  it.row0[2] = it.seg_start;
  it.len[2] = c > 0 ? seg_len : 0;
  it.pos0[2] = seg_pos0;
  item_key_tiles(it, tx_max, p.window);
  it.ok = it.total > 0;  // always, for a valid item (a token sees itself)
  return it;
}

// A work item of a forest: segment s is a node, seg_state_idx its parent's segment (-1 for a
// root).  The parent chain is walked twice (depth first, then the slots from the parent up
// to the root); a chain longer than kForestRanges - 1 or leaving the table skips the item.
__device__ __forceinline__ AttnItem<kForestRanges> attn_item_forest(const int32_t* meta, const MetaLayout& L,
                                                                    const TcParams& p, int q) {
  AttnItem<kForestRanges> it;
  const int nw = meta[H_NWORK];
  it.g = q / nw;
  const int r = q - it.g * nw;
  it.ok = 0;
  it.status = 0;
  it.total = 0;
  const int w = meta[L.work_order + r];
  if (p.checks && !attn_item_in_bounds(meta, L, w)) {
    it.status = FORK_STATUS_CHECK;
    return it;
  }
  const int s = meta[L.work_seg + w];
  it.off = meta[L.work_off + w];
  it.seg_start = meta[L.seg_start + s];
  const int seg_len = meta[L.seg_len + s];
  const int seg_pos0 = meta[L.seg_pos0 + s];
  const int tile = kRows / p.G;
  it.n_all = min(p.two_tiles ? 2 * tile : tile, seg_len - it.off);
  it.ntiles = it.n_all > tile ? 2 : 1;
  it.tx_min = seg_pos0 + it.off;
  const int tx_max = it.tx_min + it.n_all - 1;
  const int nseg = meta[H_NSEG], T = meta[H_T];
  int na = 0;
  for (int a = meta[L.seg_state_idx + s]; a >= 0; a = meta[L.seg_state_idx + a]) {
    if (na == kForestRanges - 1 || a >= nseg) {
      it.status = FORK_STATUS_BAD_DESC;
      return it;
    }
    ++na;
  }
#pragma unroll
  for (int k = 0; k < kForestRanges; ++k) {
    it.row0[k] = 0;
    it.len[k] = 0;
    it.pos0[k] = 0;
  }
  for (int k = na - 1, a = meta[L.seg_state_idx + s]; k >= 0; --k, a = meta[L.seg_state_idx + a]) {
    it.row0[k] = meta[L.seg_start + a];
    it.len[k] = meta[L.seg_len + a];
    it.pos0[k] = meta[L.seg_pos0 + a];
    if (p.checks && (it.row0[k] < 0 || it.len[k] < 0 || it.row0[k] + it.len[k] > T)) {
      it.status = FORK_STATUS_CHECK;
      return it;
    }
  }
  it.row0[na] = it.seg_start;
  it.len[na] = seg_len;
  it.pos0[na] = seg_pos0;
  item_key_tiles(it, tx_max, p.window);
  it.ok = it.total > 0;
  return it;
}

// Persistent kernel: one CTA per SM takes work items in longest-first order: item
// blockIdx.x first, then the next unclaimed one (an atomic counter, read by the producer,
// which hands each item index to the other roles through a small ring in shared memory).  TMEM, barriers and tensor-map prefetches are set up once; the
// loads run on into the next item as slots free up, and the next item's query tiles land
// while the current item's last products and output rows finish.  Barrier phases follow
// running counts (key tiles F, items, per-tile S and O), identical in every role.
template <int D, int NR>
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
  if (NR == kForestRanges && meta[H_FOREST] != 1) {  // round tables given to the forest instance
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_BAD_DESC);
    return;
  }
  const int n_items = meta[H_NWORK] * p.Hkv;
  if (static_cast<int>(blockIdx.x) >= n_items) return;
  const int G = p.G;
  const int tile = kRows / G;  // tokens per MMA tile

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::BAR + B_COUNT * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + LY::BAR + B_COUNT * 8 + 8);
  // per softmax warp: the current item's range table (first tile, tile count, length,
  // first position per slot), read in the key-tile loop instead of holding registers
  int* rtab_all = reinterpret_cast<int*>(smem + LY::BAR + B_COUNT * 8 + 16);
  // claimed work items (AttnItem, ok == 0 marks the end), written by the producer
  AttnItem<NR>* ring = reinterpret_cast<AttnItem<NR>*>(smem + LY::BAR + B_COUNT * 8 + 16 + 8 * (4 * NR) * 4);
  static_assert(B_COUNT * 8 + 16 + 8 * (4 * NR) * 4 + kItemRing * sizeof(AttnItem<NR>) <= 2048, "barrier region");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    tc::mbar_init(&bars[B_QFULL], 1);
    tc::mbar_init(&bars[B_QEMPTY], 1);
    for (int k = 0; k < 2; ++k) {
      tc::mbar_init(&bars[B_KVFULL0 + k], 1);
      tc::mbar_init(&bars[B_KEMPTY0 + k], 1);
      tc::mbar_init(&bars[B_VEMPTY0 + k], 1);
      tc::mbar_init(&bars[B_SFULL0 + k], 1);
      tc::mbar_init(&bars[B_PFULL0 + k], 128);
      tc::mbar_init(&bars[B_OFULL0 + k], 1);
      tc::mbar_init(&bars[B_OFREE0 + k], 128);
    }
    tc::mbar_init(&bars[B_FIN], 1);
    tc::mbar_init(&bars[B_QROT], 256);
    tc::mbar_init(&bars[B_STALL], 1);  // completed by nothing (FORK_TEST_STALL)
    for (int k = 0; k < kItemRing; ++k) {
      tc::mbar_init(&bars[B_ITEMF0 + k], 1);
      tc::mbar_init(&bars[B_ITEME0 + k], 9);  // the issuer and the 8 softmax warps have read it
    }
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
  auto tm_s = [&](int t) -> uint32_t { return tmem + static_cast<uint32_t>(t) * 128u; };
  auto tm_o = [&](int t) -> uint32_t { return tmem + 256u + static_cast<uint32_t>(t * D); };
  unsigned char* sQ = smem + LY::Q;
  unsigned char* sK = smem + LY::K;
  unsigned char* sV = smem + LY::V;
  // flat key-tile index f of an item -> range slot r, first key row, length, first position, tile
  struct KT {
    int r, row0, len, pos0, t;
  };
  auto key_tile = [&](const AttnItem<NR>& it, int f) -> KT {
    if constexpr (NR == kRoundRanges) {
      if (f < it.cnt[0]) return {0, it.row0[0], it.len[0], it.pos0[0], it.lo[0] + f};
      f -= it.cnt[0];
      if (f < it.cnt[1]) return {1, it.row0[1], it.len[1], it.pos0[1], it.lo[1] + f};
      f -= it.cnt[1];
      return {2, it.row0[2], it.len[2], it.pos0[2], it.lo[2] + f};
    } else {
      int r = 0;
      while (r < NR - 1 && f >= it.cnt[r]) {
        f -= it.cnt[r];
        ++r;
      }
      return {r, it.row0[r], it.len[r], it.pos0[r], it.lo[r] + f};
    }
  };

  if (warp == 1) {
    // ===================== TMA producer (lane 0) =====================
    if (lane == 0) {
      tc::prefetch_tmap(&qmap);
      tc::prefetch_tmap(&kmap);
      tc::prefetch_tmap(&vmap);
      if (p.prefix_rows > 0) {
        tc::prefetch_tmap(&pkmap);
        tc::prefetch_tmap(&pvmap);
      }
      auto wait = [&](int b, uint32_t par) -> bool { return tc::mbar_wait(&bars[b], par, abort, p.wait_ns); };
      bool ok = true;
      int F = 0, issued = 0, nq = 0, n = 0;
      for (int q = blockIdx.x;; q = static_cast<int>(gridDim.x) + atomicAdd(p.work_ctr, 1)) {
        AttnItem<NR> it;
        if (q < n_items) {
          if constexpr (NR == kRoundRanges) it = attn_item(meta, L, p, q);
          else it = attn_item_forest(meta, L, p, q);
          if (!it.ok) {  // skipped by every role: never handed on
            if (it.status) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, it.status);
            continue;
          }
        } else {
          it.ok = 0;  // the end
        }
        // hand the item to the other roles through ring slot n mod 4, free once all of
        // them have read the item four back
        const int slot = n & (kItemRing - 1);
        if (n >= kItemRing && !(ok = wait(B_ITEME0 + slot, ((n / kItemRing) - 1) & 1))) break;
        ring[slot] = it;
        tc::mbar_arrive(&bars[B_ITEMF0 + slot]);
        ++n;
        if (!it.ok) break;
        // the query tiles, once the previous item's QK^T products have read theirs
        if (nq > 0 && !(ok = wait(B_QEMPTY, (nq - 1) & 1))) break;
        tc::mbar_expect_tx(&bars[B_QFULL], it.ntiles * NB * kBox);
        for (int t = 0; t < it.ntiles; ++t)
          for (int b = 0; b < NB; ++b)
            tc::tma_load_3d(sQ + (t * NB + b) * kBox, &qmap, &bars[B_QFULL], b * 64, it.g * G,
                            it.seg_start + it.off + t * tile);
        ++nq;
        // K_F waits for the QK^T products of K_{F-2} (its slot's previous reader), V_F for
        // the PV products of V_{F-2}; both land on the slot's one barrier, whose phase also
        // needs the arrival made after both copies were issued
        for (int f = 0; f < it.total; ++f, ++F) {
          const int st = F & 1;
          const KT kt = key_tile(it, f);
          const bool pre = NR == kRoundRanges && kt.r == 0;  // a round's prefix rows
          const CUtensorMap* km = pre ? &pkmap : &kmap;
          const CUtensorMap* vm = pre ? &pvmap : &vmap;
          const int row = kt.row0 + kt.t * kKeys;
          if (F >= 2 && !(ok = wait(B_KEMPTY0 + st, ((F >> 1) - 1) & 1))) break;
          tc::mbar_expect_tx_only(&bars[B_KVFULL0 + st], NB * kBox);
          for (int b = 0; b < NB; ++b)
            tc::tma_load_3d(sK + (st * NB + b) * kBox, km, &bars[B_KVFULL0 + st], b * 64, it.g, row);
          issued = F + 1;
          const bool vok = F < 2 || wait(B_VEMPTY0 + st, ((F >> 1) - 1) & 1);
          if (vok) {
            tc::mbar_expect_tx_only(&bars[B_KVFULL0 + st], NB * kBox);
            for (int b = 0; b < NB; ++b)
              tc::tma_load_3d(sV + (st * NB + b) * kBox, vm, &bars[B_KVFULL0 + st], b * 64, it.g, row);
          }
          tc::mbar_arrive(&bars[B_KVFULL0 + st]);  // after an abort: the phase ends with the K copy
          ok = vok;
          if (!ok) break;
        }
        if (!ok) break;
      }
      // drain: the last query tiles and the last copies issued into each slot complete by
      // themselves (no copy is issued after them, so their phases are the barriers' last)
      if (nq > 0) tc::mbar_drain(&bars[B_QFULL], (nq - 1) & 1);
      for (int f = max(0, issued - 2); f < issued; ++f) tc::mbar_drain(&bars[B_KVFULL0 + (f & 1)], (f >> 1) & 1);
    }
  } else if (warp == 0) {
    // ===================== MMA issuer (lane 0 alone) =====================
    // The loop is kept short: the issuing thread shares its scheduler with two softmax
    // warps, and every instruction between two groups of products leaves the tensor
    // cores idle.  Pad rows past the stream end are zero in the value copy, so V tiles
    // need no fix-up here.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16(128, kKeys, 0, 0);
      constexpr uint32_t idesc_pv = tc::idesc_fp16(128, D, 0, 1);  // P and V fp16
      // descriptors are built once; the start-address field (16-byte units, low word) is
      // then advanced by constants: +2 per 32-byte k step, +kBox/16 per box
      const uint64_t dq = tc::sdesc_sw128(tc::smem_u32(sQ), 16, 1024);
      const uint64_t dk = tc::sdesc_sw128(tc::smem_u32(sK), 16, 1024);
      const uint64_t dv = tc::sdesc_sw128(tc::smem_u32(sV), kBox, 1024);
      constexpr uint64_t kBoxU = kBox / 16, kStageU = NB * kBox / 16;
      auto wait = [&](int b, uint32_t par) -> bool { return tc::mbar_wait(&bars[b], par, abort, p.wait_ns); };
      // O_t (+)= P_t V, V in slot vs; the first product of an item overwrites O_t
      auto issue_pv = [&](int t, bool first, int vs) {
        const uint32_t a = tm_s(t);
        const uint64_t d0 = dv + vs * kStageU;
#pragma unroll
        for (int step = 0; step < kKeys / 16; ++step)
          mma_bf16_ts(tm_o(t), a + step * 8, d0 + step * (2048 / 16), idesc_pv, (!first || step > 0) ? 1u : 0u);
      };
      auto issue_qk = [&](int t, int ks) {
        const uint64_t a0 = dq + t * NB * kBoxU, b0 = dk + ks * kStageU;
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_bf16(tm_s(t), a0 + b * kBoxU + k * 2, b0 + b * kBoxU + k * 2, idesc_qk, (b | k) ? 1u : 0u);
      };
      bool ok = !p.stall || wait(B_STALL, 0);  // FORK_TEST_STALL: runs out, nothing is issued
      int F = 0, nq = 0, nS[2] = {0, 0}, nO[2] = {0, 0};
      // PV products of tile t for the item's key tile f (V in slot vs): P_t published; the
      // first one of an item overwrites O_t, which the previous item's rows have read
      auto pv = [&](int t, int f, int vs) -> bool {
        if (!wait(B_PFULL0 + t, (nS[t] - 1) & 1)) return false;
        if (f == 0 && nO[t] > 0 && !wait(B_OFREE0 + t, (nO[t] - 1) & 1)) return false;
        tc::tc_fence_after();
        issue_pv(t, f == 0, vs);
        return true;
      };
      for (int n = 0; ok; ++n) {
        const int slot = n & (kItemRing - 1);
        if (!(ok = wait(B_ITEMF0 + slot, (n / kItemRing) & 1))) break;
        const AttnItem<NR> it = ring[slot];
        tc::mbar_arrive(&bars[B_ITEME0 + slot]);
        if (!it.ok) break;
        const int ntiles = it.ntiles, total = it.total;
        if (!(ok = wait(p.rotate_q ? B_QROT : B_QFULL, nq & 1))) break;
        ++nq;
        // per key tile f: O_0 += P_0(f-1) V(f-1), S_0 = Q_0 K(f)^T, O_1 += P_1(f-1) V(f-1),
        // S_1 = Q_1 K(f)^T.  The wait for K(f), V(f) sits after the first PV products
        // rather than after QK^T products, whose operand reads fill shared memory and slow
        // the wait.
        for (int f = 0; ok && f < total; ++f, ++F) {
          const int st = F & 1;
          for (int t = 0; ok && t < ntiles; ++t) {
            // P_t(f-1) is in the TMEM columns of S_t: the products read it before S_t is
            // rewritten (tcgen05 MMAs of one thread execute in issue order)
            if (f > 0) {
              if (!(ok = pv(t, f - 1, st ^ 1))) break;
              // V_{F-1} has no reader after the last tile's PV products: its slot is
              // released before the next QK^T products are queued behind them
              if (t == ntiles - 1) tc::mma_commit(&bars[B_VEMPTY0 + (st ^ 1)]);
            }
            if (t == 0 && !(ok = wait(B_KVFULL0 + st, (F >> 1) & 1))) break;  // K(F) and V(F)
            issue_qk(t, st);
            tc::mma_commit(&bars[B_SFULL0 + t]);
            ++nS[t];
          }
          if (ok) tc::mma_commit(&bars[B_KEMPTY0 + st]);
        }
        if (!ok) break;
        tc::mma_commit(&bars[B_QEMPTY]);  // the item's QK^T products were the last readers of Q
        const int vs = (F - 1) & 1;
        for (int t = 0; ok && t < ntiles; ++t) {
          if (!(ok = pv(t, total - 1, vs))) break;
          tc::mma_commit(&bars[B_OFULL0 + t]);
          ++nO[t];
        }
        if (ok) tc::mma_commit(&bars[B_VEMPTY0 + vs]);
      }
      // every MMA issued by this thread has completed before TMEM is released (also after
      // an abort: the products already issued finish by themselves)
      tc::mma_commit(&bars[B_FIN]);
      tc::mbar_drain(&bars[B_FIN], 0);
    }
    __syncwarp();
  } else {
    // ===================== softmax warpgroups (tile t = (warp - 2) / 4, row = tid % 128) ====
    const int t = (warp - 2) >> 2;
    int* rtab = rtab_all + (warp - 2) * (4 * NR);
    const int row = tid & 127;
    const int tok = row / G, hl = row % G;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t ts = tm_s(t) + lane_base, to = tm_o(t) + lane_base;
    const float sl2 = p.scale_log2;
    int n = 0, nq = 0, nS = 0, nO = 0;
    // the next item from the ring (ok == 0: the end); false on a failed wait
    // (forest: the item's range table goes straight to this warp's table here; the
    // previous item's key loop, its only reader, is over)
    auto fetch = [&](AttnItem<NR>& it) -> bool {
      const int slot = n & (kItemRing - 1);
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&bars[B_ITEMF0 + slot], (n / kItemRing) & 1, abort, p.wait_ns)))
        return false;
      if constexpr (NR == kRoundRanges) {
        it = ring[slot];
      } else {
        const AttnItem<NR>& rs = ring[slot];
        it.ok = rs.ok;
        it.g = rs.g;
        it.seg_start = rs.seg_start;
        it.off = rs.off;
        it.n_all = rs.n_all;
        it.ntiles = rs.ntiles;
        it.tx_min = rs.tx_min;
        it.total = rs.total;
        __syncwarp();  // every lane has finished reading the previous item's table
        if (lane < NR) {
          rtab[4 * lane] = rs.lo[lane];
          rtab[4 * lane + 1] = rs.cnt[lane];
          rtab[4 * lane + 2] = rs.len[lane];
          rtab[4 * lane + 3] = rs.pos0[lane];
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars[B_ITEME0 + slot]);
      ++n;
      return true;
    };
    // rotary embedding of an item's query tiles in shared memory, thread = row, once they
    // have landed; the products read them after every thread's fence and arrival.  The
    // row's two table rows (512 bytes each) are prefetched into L1 while the tiles load.
    auto rotate = [&](const AttnItem<NR>& it) -> bool {
      if (t < it.ntiles) {
        const int tpos = it.tx_min + t * tile + min(tok, tile - 1);
        if (tpos >> 6 < p.rope_hi_rows) {
          const char* ha = reinterpret_cast<const char*>(p.rope_hi + static_cast<int64_t>(tpos >> 6) * (D / 2));
          const char* la = reinterpret_cast<const char*>(p.rope_lo + static_cast<int64_t>(tpos & 63) * (D / 2));
#pragma unroll
          for (int o = 0; o < D * 4; o += 128) {
            asm volatile("prefetch.global.L1 [%0];" ::"l"(ha + o));
            asm volatile("prefetch.global.L1 [%0];" ::"l"(la + o));
          }
        }
      }
      const bool okq = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_QFULL], nq & 1, abort, p.wait_ns));
      ++nq;
      if (okq && t < it.ntiles && tok < min(tile, it.n_all - t * tile)) {
        const int tpos = it.tx_min + t * tile + tok;
        if (tpos >> 6 < p.rope_hi_rows) rotate_q_row<D>(sQ + t * NB * kBox, row, tpos, p.rope_hi, p.rope_lo);
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&bars[B_QROT]);
      return okq;
    };
    AttnItem<NR> cur;
    bool ok = fetch(cur);
    if (ok && cur.ok && p.rotate_q) ok = rotate(cur);
    while (ok && cur.ok) {
      const bool mine = t < cur.ntiles;
      const int n_t = mine ? min(tile, cur.n_all - t * tile) : 0;  // valid tokens of this tile
      float l = 0.f;
      if (mine) {
        if constexpr (NR == kRoundRanges) {
          __syncwarp();  // every lane has finished reading the previous item's table
          if (lane == 0) {
#pragma unroll
            for (int k = 0; k < 3; ++k) {
              rtab[4 * k] = cur.lo[k];
              rtab[4 * k + 1] = cur.cnt[k];
              rtab[4 * k + 2] = cur.len[k];
              rtab[4 * k + 3] = cur.pos0[k];
            }
          }
          __syncwarp();
        }
        const int total = cur.total;
        const int txm = cur.tx_min + t * tile;  // first position of this tile
        const int txM = txm + n_t - 1;           // last valid position of this tile
        const int tx = txm + tok;
        float m_used = -INFINITY;
        for (int f = 0; ok && f < total; ++f) {
          ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_SFULL0 + t], nS & 1, abort, p.wait_ns));
          if (!ok) break;
          ++nS;
          tc::tc_fence_after();
          float sv[kKeys];
          {
            uint32_t rawv[kKeys];
#pragma unroll
            for (int i = 0; i < kKeys / 32; ++i) tc::tmem_ld32(ts + i * 32, rawv + i * 32);
            tc::tmem_wait_ld();
#pragma unroll
            for (int cc = 0; cc < kKeys; ++cc) sv[cc] = __uint_as_float(rawv[cc]);
          }
          int len, p0, u0;
          if constexpr (NR == kRoundRanges) {
            const int c0 = rtab[1], c1 = rtab[5];
            const int r = f < c0 ? 0 : (f < c0 + c1 ? 1 : 2);
            const int fr = f - (r == 0 ? 0 : (r == 1 ? c0 : c0 + c1));
            u0 = (rtab[4 * r] + fr) * kKeys;
            len = rtab[4 * r + 2];
            p0 = rtab[4 * r + 3];
          } else {
            int r = 0, fr = f;
            while (r < NR - 1 && fr >= rtab[4 * r + 1]) {
              fr -= rtab[4 * r + 1];
              ++r;
            }
            u0 = (rtab[4 * r] + fr) * kKeys;
            len = rtab[4 * r + 2];
            p0 = rtab[4 * r + 3];
          }
          const bool need_mask = (u0 + kKeys > len) || (p0 + u0 + kKeys - 1 > txm) ||
                                 (p.window > 0 && txM - (p0 + u0) >= p.window);
          if (need_mask) {
            // key u0+cc visible iff inside the range, not after the query, inside the window
            const int lim_len = len - u0;          // cc < lim_len
            const int lim_causal = tx - p0 - u0;   // cc <= lim_causal
            const int lim_win = p.window > 0 ? tx - p0 - u0 - p.window : -0x40000000;  // cc > lim_win
#pragma unroll
            for (int cc = 0; cc < kKeys; ++cc)
              if (cc >= lim_len || cc > lim_causal || cc <= lim_win) sv[cc] = -INFINITY;
          }
          // row maximum (raw scores; the scale is positive): 8 independent chains of
          // three-input maxima
          float mx[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = sv[e];
#pragma unroll
          for (int cc = 8; cc < kKeys - 8; cc += 16)
#pragma unroll
            for (int e = 0; e < 8; ++e) mx[e] = max3(mx[e], sv[cc + e], sv[cc + 8 + e]);
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], sv[kKeys - 8 + e]);
          const float mt = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * sl2;
          const bool resc = mt > m_used + kRescale;
          const float m_new = resc ? mt : m_used;
          const float base = (m_new == -INFINITY) ? 0.f : m_new;
          const float factor = resc ? exp2f(m_used - base) : 1.f;  // 0 when nothing was accumulated
          // p = 2^(s*scale*log2e - base) as fp16 pairs (key order) into the first 64 columns
          // of S_t; the row sum adds 8 pairs per fp16 accumulator (each below 2^11), then in fp32
          float rs = 0.f;
#pragma unroll
          for (int h2 = 0; h2 < 4; ++h2) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int cc = h2 * 32 + 2 * e;
              pk[e] = exp2_pair(fmaf(sv[cc], sl2, -base), fmaf(sv[cc + 1], sl2, -base));
            }
            tc::tmem_st16(ts + h2 * 16, pk);
            uint32_t acc2[2];
#pragma unroll
            for (int a = 0; a < 2; ++a) {
              acc2[a] = pk[8 * a];
#pragma unroll
              for (int e = 1; e < 8; ++e) acc2[a] = hadd2(acc2[a], pk[8 * a + e]);
            }
            const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&acc2[0]));
            const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&acc2[1]));
            rs += (f0.x + f0.y) + (f1.x + f1.y);
          }
          l = l * factor + rs;
          m_used = m_new;
          // O_t holds the products of key tiles < f (all complete: S_t(f) was committed after
          // them) and no product writes it until P_t(f) is published; rescaled after the
          // exponentials, when the scores no longer occupy registers
          if (f >= 1 && __any_sync(0xffffffffu, factor != 1.f)) {
#pragma unroll
            for (int i = 0; i < D / 32; ++i) {
              uint32_t ov[32];
              tc::tmem_ld32(to + i * 32, ov);
              tc::tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * factor);
              tc::tmem_st32(to + i * 32, ov);
            }
          }
          tc::tmem_wait_st();
          tc::tc_fence_before();
          tc::mbar_arrive(&bars[B_PFULL0 + t]);
        }
      }
      if (!ok) break;
      // the next item's query tiles are rotated before this item's output rows are
      // written, so that its first products overlap them
      AttnItem<NR> nxt;
      if (!(ok = fetch(nxt))) break;
      if (nxt.ok && p.rotate_q && !(ok = rotate(nxt))) break;
      if (mine) {
        ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars[B_OFULL0 + t], nO & 1, abort, p.wait_ns));
        if (!ok) break;
        ++nO;
        tc::tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint16_t* orow =
            p.o + (static_cast<int64_t>(cur.seg_start + cur.off + t * tile + tok) * p.Hq + cur.g * G + hl) * D;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          uint32_t ov[32];
          tc::tmem_ld32(to + i * 32, ov);
          tc::tmem_wait_ld();
          if (tok < n_t) {
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              uint4 v4;
              v4.x = pack_bf16(__uint_as_float(ov[qq * 8 + 0]) * inv, __uint_as_float(ov[qq * 8 + 1]) * inv);
              v4.y = pack_bf16(__uint_as_float(ov[qq * 8 + 2]) * inv, __uint_as_float(ov[qq * 8 + 3]) * inv);
              v4.z = pack_bf16(__uint_as_float(ov[qq * 8 + 4]) * inv, __uint_as_float(ov[qq * 8 + 5]) * inv);
              v4.w = pack_bf16(__uint_as_float(ov[qq * 8 + 6]) * inv, __uint_as_float(ov[qq * 8 + 7]) * inv);
              *reinterpret_cast<uint4*>(orow + i * 32 + qq * 8) = v4;
            }
          }
        }
        // O_t is read: the next item's first PV products may overwrite it
        tc::tc_fence_before();
        tc::mbar_arrive(&bars[B_OFREE0 + t]);
      }
      cur = nxt;
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

// ---- host side -------------------------------------------------------------------

template <int D>
int launch_attn_tc(const AttnParams& a, const CUtensorMap* maps, int grid_x, bool two_tiles, bool forest,
                   cudaStream_t s) {
  using LY = TcLayout<D>;
  // token forests: d = 128 only (the one instance built)
  auto kern = attn_tc_kernel<D, kRoundRanges>;
  if (forest) {
    if constexpr (D == 128) kern = attn_tc_kernel<D, kForestRanges>;
    else return FORK_EINVAL;
  }
  if (cuda_rc(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM)) != FORK_OK)
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
  p.two_tiles = two_tiles ? 1 : 0;
  p.rotate_q = a.rotate_q;
  p.rope_hi = a.rope_hi;
  p.rope_lo = a.rope_lo;
  p.rope_hi_rows = a.rope_hi_rows;
  p.scale_log2 = a.scale_log2;
  p.checks = a.checks;
  p.stall = a.stall;
  p.wait_ns = a.wait_ns;
  p.work_ctr = a.work_ctr;
  // one CTA per SM over all (work item, kv head) pairs (fewer when there are fewer pairs)
  const int grid = static_cast<int>(std::min<int64_t>(static_cast<int64_t>(grid_x) * a.Hkv, sm_count()));
  kern<<<grid, kThreads, LY::SMEM, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  return cuda_rc(cudaGetLastError());
}

template int launch_attn_tc<64>(const AttnParams&, const CUtensorMap*, int, bool, bool, cudaStream_t);
template int launch_attn_tc<128>(const AttnParams&, const CUtensorMap*, int, bool, bool, cudaStream_t);

}  // namespace fork
