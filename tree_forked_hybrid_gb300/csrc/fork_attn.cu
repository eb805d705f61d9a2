// fork_attn entry point: rotary tables, key rotation, then the attention kernel.
//
// Rotary embedding (onedev summary "무엇과 다른가": a question's positions
// continue from P so it gets the rotary positions of its isolated prompt):
// pair (i, i + d/2) of a head vector at position t is rotated by the angle
// t * theta^(-2i/d).  Angles are formed in float64 on the device as
// t = 64 a + b with two small tables of (cos, sin), combined in float32 by the
// angle-addition formula.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include <cuda_fp16.h>

#include "fork_attn.cuh"

namespace fork {

static int64_t rope_hi_rows(int64_t max_pos) { return (max_pos + 128 + 63) / 64; }

// Inverse frequencies f_i = theta^(-2i/d) of the rotary embedding, formed on the host in
// fp64 (d/2 <= 64 values, passed by value)
struct RopeFreq {
  double f[64];
};

// (cos, sin) tables: hi[a][i] of the angle 64 a f_i, lo[b][i] of b f_i (b < 64); fp64
// angles and sincos, stored as fp32
__global__ void rope_tables_kernel(float2* hi, int hi_rows, float2* lo, int half, const RopeFreq freq) {
  const int64_t n_hi = static_cast<int64_t>(hi_rows) * half;
  const int64_t n = n_hi + 64 * half;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool is_hi = idx < n_hi;
    const int64_t e = is_hi ? idx : idx - n_hi;
    const int i = static_cast<int>(e % half);
    const int64_t t = is_hi ? (e / half) * 64 : e / half;
    const double ang = static_cast<double>(t) * freq.f[i];
    double sn, cs;
    sincos(ang, &sn, &cs);
    const float2 v = make_float2(static_cast<float>(cs), static_cast<float>(sn));
    if (is_hi) hi[e] = v; else lo[e] = v;
  }
}

// Rotate every row of a stream tensor [T_cap, heads, D] (position from the
// metadata) and of a prefix tensor [prefix_rows, heads, D] (position = row index
// inside its request's prefix) into the workspace.  A thread takes 8 pairs (one
// 16-byte piece of each half) of one row for every head: the pairs' (cos, sin)
// are formed once from the two tables, and the loads of 8 heads are issued before
// their rotation; a block of 256 threads covers 256 / (D / 16) rows.
template <int D>
__global__ void __launch_bounds__(256) rope_rows_kernel(const int32_t* __restrict__ meta, MetaLayout L,
                                 const uint16_t* __restrict__ k, const uint16_t* __restrict__ pk,
                                 uint16_t* __restrict__ kr, uint16_t* __restrict__ pkr,
                                 int prefix_rows, int heads, const float2* __restrict__ hi,
                                 const float2* __restrict__ lo, int hi_rows) {
  if (meta[H_VALID] == 0) return;
  constexpr int HALF = D / 2;
  constexpr int GRP = HALF / 8;  // 8-pair groups per row
  constexpr int RPB = 256 / GRP;  // rows per block
  const int T = meta[H_T];
  const int R = meta[H_R];
  const int64_t rows = static_cast<int64_t>(T) + prefix_rows;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * RPB + threadIdx.x / GRP;
  const int i0 = (threadIdx.x % GRP) * 8;
  if (row >= rows) return;
  int t;
  const uint16_t* src;
  uint16_t* dst;
  if (row < T) {
    t = meta[L.tok_pos + row];
    src = k + row * heads * D;
    dst = kr + row * heads * D;
  } else {
    const int pr = static_cast<int>(row - T);
    // request owning prefix row pr: last j with prefix_off[j] <= pr
    int a = 0, b = R;
    while (b - a > 1) {
      const int mid = (a + b) >> 1;
      if (meta[L.req_prefix_off + mid] <= pr) a = mid; else b = mid;
    }
    t = pr - meta[L.req_prefix_off + a];
    src = pk + static_cast<int64_t>(pr) * heads * D;
    dst = pkr + static_cast<int64_t>(pr) * heads * D;
  }
  if (t < 0 || (t >> 6) >= hi_rows) {
    // position beyond the rotary table: the prefix buffers given to fork_attn are
    // shorter than the descriptor's prefix lengths
    atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_BAD_PREFIX);
    return;
  }
  // (cos, sin) of pairs i0..i0+7 at position t = 64 a + b, by angle addition
  const float4* A = reinterpret_cast<const float4*>(hi + static_cast<int64_t>(t >> 6) * HALF + i0);
  const float4* B = reinterpret_cast<const float4*>(lo + static_cast<int64_t>(t & 63) * HALF + i0);
  float cs[8], sn[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 a4 = A[q], b4 = B[q];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float ac = e ? a4.z : a4.x, as = e ? a4.w : a4.y;
      const float bc = e ? b4.z : b4.x, bs = e ? b4.w : b4.y;
      cs[2 * q + e] = ac * bc - as * bs;
      sn[2 * q + e] = as * bc + ac * bs;
    }
  }
  for (int h0 = 0; h0 < heads; h0 += 8) {
    const int nh = min(8, heads - h0);
    uint4 xa[8], xb[8];
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) {
      if (hh < nh) {
        xa[hh] = *reinterpret_cast<const uint4*>(src + (h0 + hh) * D + i0);
        xb[hh] = *reinterpret_cast<const uint4*>(src + (h0 + hh) * D + i0 + HALF);
      }
    }
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) {
      if (hh >= nh) continue;
      const uint32_t aw[4] = {xa[hh].x, xa[hh].y, xa[hh].z, xa[hh].w};
      const uint32_t bw[4] = {xb[hh].x, xb[hh].y, xb[hh].z, xb[hh].w};
      uint32_t oa[4], ob[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float ya[2], yb[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float x0 = bf2f(static_cast<uint16_t>(e ? aw[q] >> 16 : aw[q] & 0xffffu));
          const float x1 = bf2f(static_cast<uint16_t>(e ? bw[q] >> 16 : bw[q] & 0xffffu));
          ya[e] = x0 * cs[2 * q + e] - x1 * sn[2 * q + e];
          yb[e] = x1 * cs[2 * q + e] + x0 * sn[2 * q + e];
        }
        oa[q] = static_cast<uint32_t>(f2bf(ya[0])) | (static_cast<uint32_t>(f2bf(ya[1])) << 16);
        ob[q] = static_cast<uint32_t>(f2bf(yb[0])) | (static_cast<uint32_t>(f2bf(yb[1])) << 16);
      }
      *reinterpret_cast<uint4*>(dst + (h0 + hh) * D + i0) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
      *reinterpret_cast<uint4*>(dst + (h0 + hh) * D + i0 + HALF) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
    }
  }
}

// blocks of rope_rows_kernel for rows_cap rows
template <int D>
static int rope_blocks(int64_t rows_cap, int heads) {
  (void)heads;
  constexpr int RPB = 256 / (D / 16);
  return static_cast<int>(std::max<int64_t>((rows_cap + RPB - 1) / RPB, 1));
}

// cuTensorMapEncodeTiled, fetched once through the runtime (no link-time
// dependency on the driver library).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D bf16 tensor [rows][heads][d] read in boxes of {box_d elements, box_heads, box_rows}
// (128-byte swizzle or none), zero fill outside the tensor.
bool encode_map_3d(CUtensorMap* m, const void* base, int d, int heads, int64_t rows, int box_d, int box_heads,
                   int box_rows, bool swizzle128) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows < 1 ? 1 : rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(heads) * d * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_d), static_cast<cuuint32_t>(box_heads),
                       static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool make_map(CUtensorMap* m, const void* base, int d, int heads, int64_t rows, int box_heads,
                     int box_rows) {
  return encode_map_3d(m, base, d, heads, rows, 64, box_heads, box_rows, true);
}

struct AttnWs {
  size_t qr, kr, pkr, hi, lo, vh, pvh, ctr, total;
};

// With the rotary embedding: rotated keys (stream, prefix), the two rotary tables and, for
// the warp-MMA kernel only, rotated queries (the tcgen05 kernel rotates its query tiles in
// shared memory).  For the tcgen05 kernel: the values as fp16 (stream, prefix), its PV
// operand (the exponentials stay fp16), and the counter of claimed work items.
static AttnWs attn_ws(int64_t T_cap, int64_t prefix_rows, int64_t Hq, int64_t Hkv, int64_t d, bool warp_mma,
                      bool rope) {
  AttnWs w;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t kv = static_cast<size_t>(T_cap) * Hkv * d * 2, pkv = static_cast<size_t>(prefix_rows) * Hkv * d * 2;
  w.qr = 0;
  w.kr = al(w.qr + (rope && warp_mma ? static_cast<size_t>(T_cap) * Hq * d * 2 : 0));
  w.pkr = al(w.kr + (rope ? kv : 0));
  w.hi = al(w.pkr + (rope ? pkv : 0));
  w.lo = al(w.hi + (rope ? static_cast<size_t>(rope_hi_rows(T_cap + prefix_rows)) * (d / 2) * 8 : 0));
  w.vh = al(w.lo + (rope ? static_cast<size_t>(64) * (d / 2) * 8 : 0));
  w.pvh = al(w.vh + (warp_mma ? 0 : kv));
  w.ctr = al(w.pvh + (warp_mma ? 0 : pkv));
  w.total = al(w.ctr + (warp_mma ? 0 : 4));
  return w;
}

// Values of the stream rows [0, T) and of the prefix rows as fp16 (8 elements per thread);
// also zeroes the counter through which the attention kernel's CTAs claim work items.
// The rows [T, min(T_cap, T + 128)) of the copy are set to zero: a key tile that starts
// inside the stream reads at most 127 rows past its range, and rows past T are not the
// caller's data (any bits), while the products need finite values there (p = 0 and
// 0 * NaN is not 0).  Rows past T_cap read as zero from the tensor map.
__global__ void __launch_bounds__(256) v_half_kernel(const int32_t* __restrict__ meta, const uint16_t* __restrict__ v,
                                                     const uint16_t* __restrict__ pv, uint16_t* __restrict__ vh,
                                                     uint16_t* __restrict__ pvh, int64_t row_elems, int prefix_rows,
                                                     int T_cap, int* __restrict__ work_ctr) {
  if (blockIdx.x == 0 && threadIdx.x == 0) *work_ctr = 0;  // the attention kernel's item counter
  if (meta[H_VALID] == 0) return;
  const int T = meta[H_T];
  const int64_t n_stream = static_cast<int64_t>(T) * row_elems / 8;
  const int64_t n_zero = n_stream + static_cast<int64_t>(min(T_cap, T + 128) - T) * row_elems / 8;
  const int64_t n_all = n_zero + static_cast<int64_t>(prefix_rows) * row_elems / 8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n_all;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (i >= n_stream && i < n_zero) {
      reinterpret_cast<uint4*>(vh)[i] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const bool st = i < n_stream;
    const uint4 x = st ? reinterpret_cast<const uint4*>(v)[i] : reinterpret_cast<const uint4*>(pv)[i - n_zero];
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half2 hh = __floats2half2_rn(bf2f(static_cast<uint16_t>(w[e] & 0xffffu)), bf2f(static_cast<uint16_t>(w[e] >> 16)));
      o[e] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    const uint4 y = make_uint4(o[0], o[1], o[2], o[3]);
    if (st) reinterpret_cast<uint4*>(vh)[i] = y; else reinterpret_cast<uint4*>(pvh)[i - n_zero] = y;
  }
}

}  // namespace fork

using namespace fork;

extern "C" size_t fork_attn_workspace_bytes(int32_t T_cap, int32_t prefix_rows, int32_t Hq,
                                            int32_t Hkv, int32_t d, float rope_theta, uint32_t flags) {
  if (T_cap < 1 || prefix_rows < 0 || Hkv < 1 || Hq < Hkv || (d != 64 && d != 128)) return 0;
  return attn_ws(T_cap, prefix_rows, Hq, Hkv, d, (flags & FORK_WARP_MMA) != 0, rope_theta != 0.f).total;
}

extern "C" int fork_attn(const fork_meta* m, const uint16_t* q, const uint16_t* k,
                         const uint16_t* v, uint16_t* o, int32_t Hq, int32_t Hkv, int32_t d,
                         int32_t window, float rope_theta, float scale, const uint16_t* prefix_k,
                         const uint16_t* prefix_v, int32_t prefix_rows, void* workspace,
                         size_t ws_bytes, uint32_t flags, void* stream) {
  MetaLayout L;
  int rc = check_meta(m, &L);
  if (rc != FORK_OK) return rc;
  if (!q || !k || !v || !o) return FORK_EINVAL;
  if (!is_aligned16(q) || !is_aligned16(k) || !is_aligned16(v) || !is_aligned16(o)) return FORK_EINVAL;
  if (d != 64 && d != 128) return FORK_EINVAL;
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv != 0) return FORK_EINVAL;
  const int G = Hq / Hkv;
  // a work item is one 128-row query tile, or two for the tcgen05 kernel
  const bool warp_mma = (flags & FORK_WARP_MMA) != 0;
  if (G * m->tile_tokens != 128 && (warp_mma || G * m->tile_tokens != 256)) return FORK_EINVAL;
  if (window < 0 || prefix_rows < 0 || !(scale > 0.f) || !std::isfinite(scale)) return FORK_EINVAL;
  if (!(rope_theta >= 0.f) || !std::isfinite(rope_theta)) return FORK_EINVAL;
  if (prefix_rows > 0 && (!prefix_k || !prefix_v || !is_aligned16(prefix_k) || !is_aligned16(prefix_v)))
    return FORK_EINVAL;
  // token forests: the tcgen05 kernel's forest instance (d = 128), every key in the stream
  const bool forest = (flags & FORK_FOREST) != 0;
  if (forest && (d != 128 || warp_mma || prefix_rows != 0 || prefix_k || prefix_v)) return FORK_EINVAL;
  if ((rc = check_device()) != FORK_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  AttnParams p;
  p.meta = static_cast<const int32_t*>(m->d_buf);
  p.L = L;
  p.q = q;
  p.k = k;
  p.v = v;
  p.prefix_k = prefix_k;
  p.prefix_v = prefix_v;
  p.o = o;
  p.rope_hi = nullptr;
  p.rope_lo = nullptr;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.prefix_rows = prefix_k ? prefix_rows : 0;
  p.window = window;
  p.rope_theta = rope_theta;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.rope_hi_rows = 0;
  p.rotate_q = 0;
  p.checks = (flags & FORK_CHECKS) ? 1 : 0;
  p.stall = (flags & FORK_TEST_STALL) ? 1 : 0;
  p.wait_ns = wait_ns_of(m);
  p.work_ctr = nullptr;

  const AttnWs w = attn_ws(L.T_cap, prefix_rows, Hq, Hkv, d, warp_mma, rope_theta != 0.f);
  if (w.total > 0 && (!workspace || ws_bytes < w.total || !is_aligned16(workspace))) return FORK_EINVAL;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  if (rope_theta != 0.f) {
    uint16_t* qr = reinterpret_cast<uint16_t*>(ws + w.qr);
    uint16_t* kr = reinterpret_cast<uint16_t*>(ws + w.kr);
    uint16_t* pkr = reinterpret_cast<uint16_t*>(ws + w.pkr);
    float2* hi = reinterpret_cast<float2*>(ws + w.hi);
    float2* lo = reinterpret_cast<float2*>(ws + w.lo);
    const int hi_rows = static_cast<int>(rope_hi_rows(static_cast<int64_t>(L.T_cap) + prefix_rows));
    RopeFreq freq;
    for (int i = 0; i < 64; ++i) freq.f[i] = i < d / 2 ? std::pow(static_cast<double>(rope_theta), -2.0 * i / d) : 0.0;
    rope_tables_kernel<<<2 * sm_count(), 128, 0, s>>>(hi, hi_rows, lo, d / 2, freq);
    // keys of the stream and of the prefix (grids from the capacities: blocks past the
    // round's rows return); the queries here only for the warp-MMA kernel: the tcgen05
    // kernel rotates each query tile in shared memory once it has landed
    const int64_t krows = static_cast<int64_t>(L.T_cap) + prefix_rows;
    if (d == 64) {
      rope_rows_kernel<64><<<rope_blocks<64>(krows, Hkv), 256, 0, s>>>(p.meta, L, k, prefix_k, kr, pkr, prefix_rows,
                                                                        Hkv, hi, lo, hi_rows);
      if (warp_mma)
        rope_rows_kernel<64><<<rope_blocks<64>(L.T_cap, Hq), 256, 0, s>>>(p.meta, L, q, nullptr, qr, nullptr, 0, Hq,
                                                                           hi, lo, hi_rows);
    } else {
      rope_rows_kernel<128><<<rope_blocks<128>(krows, Hkv), 256, 0, s>>>(p.meta, L, k, prefix_k, kr, pkr, prefix_rows,
                                                                          Hkv, hi, lo, hi_rows);
      if (warp_mma)
        rope_rows_kernel<128><<<rope_blocks<128>(L.T_cap, Hq), 256, 0, s>>>(p.meta, L, q, nullptr, qr, nullptr, 0,
                                                                             Hq, hi, lo, hi_rows);
    }
    if (warp_mma) p.q = qr;
    p.k = kr;
    p.prefix_k = pkr;
    p.rope_hi = hi;
    p.rope_lo = lo;
    p.rope_hi_rows = hi_rows;
    p.rotate_q = warp_mma ? 0 : 1;
    p.rope_theta = 0.f;  // keys rotated; queries rotated above or by the attention kernel
  }
  const uint16_t* vtc = v;  // values read by the tcgen05 kernel: fp16 copies
  const uint16_t* pvtc = prefix_v;
  if (!warp_mma) {
    uint16_t* vh = reinterpret_cast<uint16_t*>(ws + w.vh);
    uint16_t* pvh = reinterpret_cast<uint16_t*>(ws + w.pvh);
    const int64_t row_elems = static_cast<int64_t>(Hkv) * d;
    const int64_t n8 = (static_cast<int64_t>(L.T_cap) + p.prefix_rows) * row_elems / 8;
    const int blocks = static_cast<int>(std::min<int64_t>((n8 + 255) / 256, 8 * sm_count()));
    p.work_ctr = reinterpret_cast<int*>(ws + w.ctr);
    v_half_kernel<<<std::max(blocks, 1), 256, 0, s>>>(p.meta, v, prefix_v, vh, pvh, row_elems, p.prefix_rows,
                                                      L.T_cap, p.work_ctr);
    vtc = vh;
    pvtc = pvh;
  }
  if (cuda_rc(cudaGetLastError()) != FORK_OK) return FORK_ECUDA;
  const int grid_x = static_cast<int>(std::min<int64_t>(
      L.max_work, (L.T_cap + m->tile_tokens - 1) / m->tile_tokens + L.max_seg));
  if (warp_mma)
    return d == 64 ? launch_attn_mma<64>(p, grid_x, s) : launch_attn_mma<128>(p, grid_x, s);
  alignas(128) CUtensorMap maps[5];
  const uint16_t* pk = p.prefix_rows > 0 ? p.prefix_k : p.k;
  const uint16_t* pv = p.prefix_rows > 0 ? pvtc : vtc;
  const int prow = p.prefix_rows > 0 ? p.prefix_rows : L.T_cap;
  const bool two = G * m->tile_tokens == 256;
  const int tile = 128 / G;  // tokens of one 128-row query tile
  if (!make_map(&maps[0], p.q, d, Hq, L.T_cap, G, tile) ||
      !make_map(&maps[1], p.k, d, Hkv, L.T_cap, 1, 128) || !make_map(&maps[2], vtc, d, Hkv, L.T_cap, 1, 128) ||
      !make_map(&maps[3], pk, d, Hkv, prow, 1, 128) || !make_map(&maps[4], pv, d, Hkv, prow, 1, 128))
    return FORK_ECUDA;
  return d == 64 ? launch_attn_tc<64>(p, maps, grid_x, two, forest, s)
                 : launch_attn_tc<128>(p, maps, grid_x, two, forest, s);
}

// ---- fork_attn_noalloc: fork_attn with the library's own scratch area -------------
//
// Some callers cannot allocate device memory at all: they only hold pointers to
// their inputs and outputs (for example a host runtime that plans every device
// buffer up front and forbids allocation inside its serving loop, since
// cudaMalloc and cudaFree synchronise the device).  For them the scratch that
// fork_attn needs (rotated keys and rotary tables) lives in this file-scope
// device array instead of a caller workspace.  The module that holds it is loaded
// on each GPU that uses the library, and the array stays allocated there until
// the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FORK_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};  // device address of the array, per device
}  // namespace

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once per
// device with that device current (this also loads the module on that device).
static int noalloc_scratch(void** out) {
  int dev = 0;
  if (cuda_rc(cudaGetDevice(&dev)) != FORK_OK) return FORK_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return FORK_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cuda_rc(cudaGetSymbolAddress(&p, g_noalloc_scratch)) != FORK_OK || p == nullptr) return FORK_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return FORK_OK;
}

extern "C" int fork_attn_noalloc(const fork_meta* m, const uint16_t* q, const uint16_t* k,
                                 const uint16_t* v, uint16_t* o, int32_t Hq, int32_t Hkv, int32_t d,
                                 int32_t window, float rope_theta, float scale,
                                 const uint16_t* prefix_k, const uint16_t* prefix_v,
                                 int32_t prefix_rows, uint32_t flags, void* stream) {
  MetaLayout L;
  int rc = check_meta(m, &L);
  if (rc != FORK_OK) return rc;
  if (prefix_rows < 0 || Hkv < 1 || (d != 64 && d != 128)) return FORK_EINVAL;
  const size_t need = fork_attn_workspace_bytes(L.T_cap, prefix_rows, Hq, Hkv, d, rope_theta, flags);
  if (need > FORK_NOALLOC_SCRATCH_BYTES) return FORK_ECAPACITY;
  void* scratch = nullptr;
  if (need > 0 && (rc = noalloc_scratch(&scratch)) != FORK_OK) return rc;
  return fork_attn(m, q, k, v, o, Hq, Hkv, d, window, rope_theta, scale, prefix_k, prefix_v, prefix_rows,
                   scratch, need > 0 ? FORK_NOALLOC_SCRATCH_BYTES : 0, flags, stream);
}
