// Tree-masked GQA attention on CUDA cores: the path for fp32 and for shapes whose
// node x group rows do not fill a tensor-core tile (or whose head_dim the tile kernel
// does not take).
//
// PTD §3.1: node i attends to the committed prefix and to its observable set pi(i)
// = {i} U pi(parent(i)).  One warp owns one (b, h, i) query row: each lane scores one
// visible key per step (full dot product over D), the warp keeps an online softmax
// (running max / sum) and accumulates sum_j p_j v_j with lanes split over D.
#include "tv_kernels.cuh"

namespace tv {

constexpr int kSimtWarps = 4;
constexpr int kSimtMaxD = 256;

template <typename T>
__device__ __forceinline__ float ldx(const T* p, size_t i) {
  if constexpr (sizeof(T) == 2)
    return bf16_to_f32(reinterpret_cast<const uint16_t*>(p)[i]);
  else
    return p[i];
}

template <typename T>
__device__ __forceinline__ void stx(T* p, size_t i, float v) {
  if constexpr (sizeof(T) == 2)
    reinterpret_cast<uint16_t*>(p)[i] = f32_to_bf16_rn(v);
  else
    p[i] = v;
}

template <typename T, int kDPL>  // kDPL = D / 32 output dims per lane
__global__ void __launch_bounds__(kSimtWarps * 32) attn_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                                   const T* __restrict__ v, T* __restrict__ out,
                                                                   const int32_t* __restrict__ parent, int B, int Hq,
                                                                   int Hkv, int D, int P, int N, int S, float scale,
                                                                   int32_t* dev_status) {
  __shared__ float s_q[kSimtWarps][kSimtMaxD];
  __shared__ int s_anc[kSimtWarps][kMaxNodes];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kSimtWarps + warp;
  const long long rows = (long long)B * Hq * N;
  if (row >= rows) return;
  const int i = (int)(row % N);
  const int h = (int)((row / N) % Hq);
  const int b = (int)(row / ((long long)N * Hq));
  const int G = Hq / Hkv;
  const int kh = h / G;
  const int32_t* par = parent + (size_t)b * N;
  // ancestors of i (root ... i), validated: each step must go to a smaller index
  int na = 0;
  if (lane == 0) {
    int a = i, cnt = 0;
    bool ok = true;
    while (a >= 0) {
      s_anc[warp][cnt++] = a;
      const int pa = par[a];
      if (!(pa < a) || (a == 0 && pa != -1) || (a > 0 && pa < 0)) {
        ok = false;
        break;
      }
      a = pa;
    }
    if (!ok) {
      set_dev_status(dev_status, TV_DEV_BAD_TREE);
      cnt = 1;
      s_anc[warp][0] = i;
    }
    na = cnt;
  }
  na = __shfl_sync(0xffffffffu, na, 0);
  const size_t qoff = (((size_t)b * Hq + h) * N + i) * D;
  for (int d = lane; d < D; d += 32) s_q[warp][d] = ldx(q, qoff + d);
  __syncwarp();
  const size_t kvbase = ((size_t)b * Hkv + kh) * (size_t)S * D;
  const int total = P + na;
  float m = -INFINITY, l = 0.f;
  float acc[kDPL];
#pragma unroll
  for (int t = 0; t < kDPL; ++t) acc[t] = 0.f;
  for (int j0 = 0; j0 < total; j0 += 32) {
    const int j = j0 + lane;
    int krow = 0;
    float s = -INFINITY;
    if (j < total) {
      krow = j < P ? j : P + s_anc[warp][j - P];
      const T* kr = k + kvbase + (size_t)krow * D;
      // eight independent partial dot products, so that the row's loads overlap
      float dot[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) dot[u] = 0.f;
      for (int d0 = 0; d0 < D; d0 += 8)
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (d0 + u < D) dot[u] = fmaf(s_q[warp][d0 + u], ldx(kr, d0 + u), dot[u]);
      s = (((dot[0] + dot[1]) + (dot[2] + dot[3])) + ((dot[4] + dot[5]) + (dot[6] + dot[7]))) * scale;
    }
    const float mnew = fmaxf(m, warp_max(s));
    const float corr = exp2f((m - mnew) * kLog2e);
    const float p = j < total ? exp2f((s - mnew) * kLog2e) : 0.f;
    l = l * corr + warp_sum(p);
#pragma unroll
    for (int t = 0; t < kDPL; ++t) acc[t] *= corr;
    const int cnt = min(32, total - j0);
    for (int jb = 0; jb < cnt; jb += 4) {
      // four value rows at a time: all their loads are issued before the FMAs
      float vv[4][kDPL], pj[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int jj = min(jb + u, cnt - 1);
        pj[u] = jb + u < cnt ? __shfl_sync(0xffffffffu, p, jj) : 0.f;
        const int rj = __shfl_sync(0xffffffffu, krow, jj);
        const T* vr = v + kvbase + (size_t)rj * D;
#pragma unroll
        for (int t = 0; t < kDPL; ++t) vv[u][t] = lane + 32 * t < D ? ldx(vr, lane + 32 * t) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int t = 0; t < kDPL; ++t) acc[t] = fmaf(pj[u], vv[u][t], acc[t]);
    }
    m = mnew;
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int t = 0; t < kDPL; ++t) stx(out, qoff + lane + 32 * t, acc[t] * inv);
}

template <typename T>
static void launch_simt_t(const void* q, const void* k, const void* v, void* out, const int32_t* parent, int B,
                          int Hq, int Hkv, int D, int P, int N, int S, float scale, int32_t* dev_status,
                          cudaStream_t stream) {
  const long long rows = (long long)B * Hq * N;
  const unsigned grid = (unsigned)((rows + kSimtWarps - 1) / kSimtWarps);
  const T* qq = reinterpret_cast<const T*>(q);
  const T* kk = reinterpret_cast<const T*>(k);
  const T* vv = reinterpret_cast<const T*>(v);
  T* oo = reinterpret_cast<T*>(out);
  switch (D / 32) {
#define TV_SIMT_CASE(n)                                                                                        \
  case n:                                                                                                      \
    attn_simt_kernel<T, n><<<grid, kSimtWarps * 32, 0, stream>>>(qq, kk, vv, oo, parent, B, Hq, Hkv, D, P, N, S, \
                                                                 scale, dev_status);                           \
    break;
    TV_SIMT_CASE(1)
    TV_SIMT_CASE(2)
    TV_SIMT_CASE(3)
    TV_SIMT_CASE(4)
    TV_SIMT_CASE(5)
    TV_SIMT_CASE(6)
    TV_SIMT_CASE(7)
    TV_SIMT_CASE(8)
#undef TV_SIMT_CASE
    default:
      break;
  }
}

cudaError_t launch_attn_simt(const void* q, const void* k, const void* v, void* out, const int32_t* parent,
                             int B, int Hq, int Hkv, int D, int P, int N, int S, float scale, tv_dtype dtype,
                             int32_t* dev_status, cudaStream_t stream) {
  if (dtype == TV_BF16)
    launch_simt_t<uint16_t>(q, k, v, out, parent, B, Hq, Hkv, D, P, N, S, scale, dev_status, stream);
  else
    launch_simt_t<float>(q, k, v, out, parent, B, Hq, Hkv, D, P, N, S, scale, dev_status, stream);
  return cudaGetLastError();
}

}  // namespace tv
