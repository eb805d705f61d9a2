// Selective options readout, eq. (1) of the Flide pages (onedev summary
// "어떻게 동작하나"; rainbus summary "前置知识"):
//     p_i(o) = exp(w_o . h_i) / sum_{o' in O_i} exp(w_o' . h_i),
// with h_i the hidden row of question i's last stream token (metadata q_last).
// One CTA per question; each warp owns options, each lane a fixed strided set
// of the D elements, reductions in a fixed tree: results do not depend on
// the rest of the round.
#include "fork_common.cuh"

namespace fork {

__global__ void __launch_bounds__(256) readout_kernel(const int32_t* __restrict__ meta, MetaLayout L,
                                                      const uint16_t* __restrict__ h, int D,
                                                      const uint16_t* __restrict__ w,
                                                      const int32_t* __restrict__ off,
                                                      float* __restrict__ p, int checks) {
  if (meta[H_VALID] == 0) return;
  const int i = blockIdx.x;
  if (i >= meta[H_NQ]) return;
  const int a = off[i], b = off[i + 1];
  const int x = meta[L.q_last + i];
  // FORK_CHECKS: offsets start at 0 and grow (at least one option each); the row is a stream row
  if (checks && (a < 0 || b <= a || (i == 0 && a != 0) || x < 0 || x >= meta[H_T])) {
    if (threadIdx.x == 0) atomicOr(const_cast<int32_t*>(meta) + H_STATUS, FORK_STATUS_CHECK);
    return;
  }
  const uint4* hrow = reinterpret_cast<const uint4*>(h + static_cast<int64_t>(x) * D);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = D / 8;
  for (int o = a + warp; o < b; o += blockDim.x / 32) {
    const uint4* wrow = reinterpret_cast<const uint4*>(w + static_cast<int64_t>(o) * D);
    float acc = 0.f;
    for (int u = lane; u < nvec; u += 32) {
      const uint4 hv = hrow[u], wv = wrow[u];
      const uint32_t hh[4] = {hv.x, hv.y, hv.z, hv.w}, ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc += bf2f(static_cast<uint16_t>(hh[e] & 0xffffu)) * bf2f(static_cast<uint16_t>(ww[e] & 0xffffu));
        acc += bf2f(static_cast<uint16_t>(hh[e] >> 16)) * bf2f(static_cast<uint16_t>(ww[e] >> 16));
      }
    }
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) p[o] = acc;  // logit
  }
  __syncthreads();
  // softmax over the question's options (warp 0; fixed order)
  if (warp == 0) {
    float mx = -INFINITY;
    for (int o = a + lane; o < b; o += 32) mx = fmaxf(mx, p[o]);
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    float sum = 0.f;
    for (int o = a + lane; o < b; o += 32) sum += expf(p[o] - mx);
    for (int s = 16; s > 0; s >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, s);
    const float inv = 1.f / sum;
    __syncwarp();
    for (int o = a + lane; o < b; o += 32) p[o] = expf(p[o] - mx) * inv;
  }
}

}  // namespace fork

using namespace fork;

extern "C" int fork_readout(const fork_meta* m, const uint16_t* h, int32_t D, const uint16_t* w_opt,
                            const int32_t* opt_off, float* p, uint32_t flags, void* stream) {
  MetaLayout L;
  int rc = check_meta(m, &L);
  if (rc != FORK_OK) return rc;
  if (!h || !w_opt || !opt_off || !p) return FORK_EINVAL;
  if (D < 8 || D % 8 != 0 || D > 16384) return FORK_EINVAL;
  if (!is_aligned16(h) || !is_aligned16(w_opt)) return FORK_EINVAL;
  if ((rc = check_device()) != FORK_OK) return rc;
  if (m->max_q == 0) return FORK_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  readout_kernel<<<m->max_q, 256, 0, s>>>(static_cast<const int32_t*>(m->d_buf), L, h, D, w_opt,
                                         opt_off, p, (flags & FORK_CHECKS) ? 1 : 0);
  return cuda_rc(cudaGetLastError());
}
