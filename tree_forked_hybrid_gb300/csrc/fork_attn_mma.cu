// Fork-masked varlen attention, legacy warp-MMA (mma.sync m16n8k16 bf16) path.
//
// Visibility (rainbus summary "方法步骤详情" step 2; onedev "무엇과 다른가"):
// key y is visible to query x iff j_y = j_x, c_y in {0, c_x}, t_y <= t_x and,
// for a sliding-window layer, t_x - t_y < W.  For one query tile (one
// segment) that is at most three contiguous key ranges: the request's prefix
// rows held outside the stream (incremental resume), its trunk segment, and
// for a question its own branch.  Inside a range, key u (position p0 + u) is
// visible to query position t iff u < len, p0 + u <= t and (W == 0 or
// t - p0 - u < W).  Rotary positions are the isolated ones (questions
// continue from P).
//
// Tiles are aligned to the segment (queries) and to each range's start
// (keys), so every output is computed in the same order whatever else the
// round contains.
#include "fork_attn.cuh"

namespace fork {

namespace {

constexpr int kRows = 128;  // query rows per CTA (tokens x grouped heads)
constexpr int kKeys = 64;   // keys per tile
constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int D>
struct Smem {
  static constexpr int LD = D + 8;  // padded row (bf16 elements): conflict-free ldmatrix
  uint16_t q[kRows * LD];
  uint16_t k[2][kKeys * LD];
  uint16_t v[2][kKeys * LD];
};

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_mma_kernel(const AttnParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem<D>& sm = *reinterpret_cast<Smem<D>*>(smem_raw);
  constexpr int LD = Smem<D>::LD;

  const int32_t* meta = p.meta;
  const MetaLayout& L = p.L;
  if (meta[H_VALID] == 0) return;
  if (static_cast<int>(blockIdx.x) >= meta[H_NWORK]) return;
  const int w = meta[L.work_order + blockIdx.x];  // longest items first
  const int g = blockIdx.y;  // kv head
  const int G = p.G;
  const int tile = kRows / G;
  if (p.checks && !attn_item_in_bounds(meta, L, w)) {
    if (threadIdx.x == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_CHECK);
    return;
  }

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

  // ---- key ranges -----------------------------------------------------------
  KeyRange rng[3];
  int nr = 0;
  const int pl = meta[L.req_prefix_len + j];
  if (pl > 0) {
    const int poff = meta[L.req_prefix_off + j];
    if (poff + pl > p.prefix_rows) {
      // the caller's prefix buffers do not hold this request's rows
      if (threadIdx.x == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_BAD_PREFIX);
      return;
    }
    rng[nr++] = {p.prefix_k, p.prefix_v, poff, pl, 0};
  }
  rng[nr++] = {p.k, p.v, meta[L.seg_trunk_start + s], meta[L.seg_trunk_len + s], pl};
  if (c > 0) rng[nr++] = {p.k, p.v, seg_start, seg_len, seg_pos0};
  int lo[3], cnt[3], total = 0;
  for (int r = 0; r < nr; ++r) {
    const int umax = min(rng[r].len - 1, tx_max - rng[r].pos0);
    int umin = 0;
    if (p.window > 0) umin = max(0, tx_min - p.window + 1 - rng[r].pos0);
    if (umax < umin) {
      lo[r] = 0;
      cnt[r] = 0;
    } else {
      lo[r] = umin / kKeys;
      cnt[r] = umax / kKeys - lo[r] + 1;
    }
    total += cnt[r];
  }

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  // ---- Q tile: rows r = token * G + grouped head ------------------------------
  {
    constexpr int CPR = D / 8;  // 16-byte chunks per row
    for (int idx = tid; idx < kRows * CPR; idx += kThreads) {
      const int r = idx / CPR, ch = idx % CPR;
      const int tok = r / G, hl = r % G;
      const bool valid = tok < n;
      const int64_t row = static_cast<int64_t>(seg_start + off + (valid ? tok : 0)) * p.Hq + g * G + hl;
      cp_async16(&sm.q[r * LD + ch * 8], p.q + row * D + ch * 8, valid);
    }
    cp_async_commit();
  }

  auto key_tile = [&](int f, int& r, int& t) {
    r = 0;
    while (r < nr && f >= cnt[r]) {
      f -= cnt[r];
      ++r;
    }
    t = lo[r] + f;
  };
  auto load_kv = [&](int f, int buf) {
    int r, t;
    key_tile(f, r, t);
    const KeyRange& kr = rng[r];
    constexpr int CPR = D / 8;
    for (int idx = tid; idx < kKeys * CPR; idx += kThreads) {
      const int u = idx / CPR, ch = idx % CPR;
      const int ku = t * kKeys + u;
      const bool valid = ku < kr.len;
      const int64_t row = static_cast<int64_t>(kr.row0 + (valid ? ku : 0)) * p.Hkv + g;
      cp_async16(&sm.k[buf][u * LD + ch * 8], kr.k + row * D + ch * 8, valid);
      cp_async16(&sm.v[buf][u * LD + ch * 8], kr.v + row * D + ch * 8, valid);
    }
    cp_async_commit();
  };

  if (total > 0) load_kv(0, 0);
  cp_async_wait<0>();
  __syncthreads();

  // Q fragments of this warp's 16 rows
  uint32_t qf[D / 16][4];
  {
    const int mi = lane >> 3, rr = (mi & 1) * 8 + (lane & 7), cc = (mi >> 1) * 8;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
      ldsm_x4(qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], &sm.q[(warp * 16 + rr) * LD + ks * 16 + cc]);
  }

  const int gq = lane >> 2, tq = lane & 3;
  const int row0 = warp * 16 + gq, row1 = row0 + 8;
  const int tpos0 = tx_min + row0 / G, tpos1 = tx_min + row1 / G;
  float o_acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float sl2 = p.scale_log2;

  for (int f = 0; f < total; ++f) {
    const int buf = f & 1;
    if (f + 1 < total) {
      load_kv(f + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    int r, t;
    key_tile(f, r, t);
    const KeyRange kr = rng[r];
    const uint16_t* sk = sm.k[buf];
    const uint16_t* sv = sm.v[buf];

    float sacc[kKeys / 8][4];
#pragma unroll
    for (int i = 0; i < kKeys / 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
    {
      const int mi = lane >> 3, kr8 = (mi >> 1) * 8 + (lane & 7), kc = (mi & 1) * 8;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < kKeys / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(b0, b1, b2, b3, &sk[(np * 16 + kr8) * LD + ks * 16 + kc]);
          mma_bf16(sacc[2 * np], qf[ks], b0, b1);
          mma_bf16(sacc[2 * np + 1], qf[ks], b2, b3);
        }
      }
    }
    // mask, scale (log2 domain) and row maxima
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < kKeys / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int u = t * kKeys + nt * 8 + 2 * tq + e;
        const int ty = kr.pos0 + u;
        const bool ok = u < kr.len;
        const bool v0 = ok && ty <= tpos0 && (p.window == 0 || tpos0 - ty < p.window);
        const bool v1 = ok && ty <= tpos1 && (p.window == 0 || tpos1 - ty < p.window);
        sacc[nt][e] = v0 ? sacc[nt][e] * sl2 : -INFINITY;
        sacc[nt][2 + e] = v1 ? sacc[nt][2 + e] * sl2 : -INFINITY;
        mx0 = fmaxf(mx0, sacc[nt][e]);
        mx1 = fmaxf(mx1, sacc[nt][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
    const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
    const float corr0 = exp2f(m0 - base0), corr1 = exp2f(m1 - base1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
    uint32_t pf[kKeys / 16][4];
#pragma unroll
    for (int nt = 0; nt < kKeys / 8; ++nt) {
      const float p00 = exp2f(sacc[nt][0] - base0), p01 = exp2f(sacc[nt][1] - base0);
      const float p10 = exp2f(sacc[nt][2] - base1), p11 = exp2f(sacc[nt][3] - base1);
      rs0 += p00 + p01;
      rs1 += p10 + p11;
      pf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p00, p01);
      pf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p10, p11);
    }
    rs0 += __shfl_xor_sync(0xffffffffu, rs0, 1);
    rs0 += __shfl_xor_sync(0xffffffffu, rs0, 2);
    rs1 += __shfl_xor_sync(0xffffffffu, rs1, 1);
    rs1 += __shfl_xor_sync(0xffffffffu, rs1, 2);
    l0 = l0 * corr0 + rs0;
    l1 = l1 * corr1 + rs1;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o_acc[i][0] *= corr0;
      o_acc[i][1] *= corr0;
      o_acc[i][2] *= corr1;
      o_acc[i][3] *= corr1;
    }
    // O += P V
    {
      const int mi = lane >> 3, vr = (mi & 1) * 8 + (lane & 7), vc = (mi >> 1) * 8;
#pragma unroll
      for (int ks = 0; ks < kKeys / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(b0, b1, b2, b3, &sv[(ks * 16 + vr) * LD + np * 16 + vc]);
          mma_bf16(o_acc[2 * np], pf[ks], b0, b1);
          mma_bf16(o_acc[2 * np + 1], pf[ks], b2, b3);
        }
      }
    }
    __syncthreads();
  }

  // ---- normalise and store ----------------------------------------------------
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int tok0 = row0 / G, hl0 = row0 % G, tok1 = row1 / G, hl1 = row1 % G;
  uint16_t* o0 = p.o + (static_cast<int64_t>(seg_start + off + tok0) * p.Hq + g * G + hl0) * D;
  uint16_t* o1 = p.o + (static_cast<int64_t>(seg_start + off + tok1) * p.Hq + g * G + hl1) * D;
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) {
    const int col = nt * 8 + 2 * tq;
    if (tok0 < n)
      *reinterpret_cast<uint32_t*>(o0 + col) = pack_bf16(o_acc[nt][0] * inv0, o_acc[nt][1] * inv0);
    if (tok1 < n)
      *reinterpret_cast<uint32_t*>(o1 + col) = pack_bf16(o_acc[nt][2] * inv1, o_acc[nt][3] * inv1);
  }
}

template <int D>
int launch_attn_mma(const AttnParams& p, int grid_x, cudaStream_t s) {
  const size_t smem = sizeof(Smem<D>);
  if (cuda_rc(cudaFuncSetAttribute(attn_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem))) != FORK_OK)
    return FORK_ECUDA;
  dim3 grid(grid_x, p.Hkv);
  attn_mma_kernel<D><<<grid, kThreads, smem, s>>>(p);
  return cuda_rc(cudaGetLastError());
}

template int launch_attn_mma<64>(const AttnParams&, int, cudaStream_t);
template int launch_attn_mma<128>(const AttnParams&, int, cudaStream_t);

}  // namespace fork
