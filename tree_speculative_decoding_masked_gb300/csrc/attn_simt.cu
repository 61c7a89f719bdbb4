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

// One CTA per (b, kv head, block of kRowsCta query rows of that head's G x N rows).
// Keys are walked in tiles of 32: the CTA stages the tile's K and V rows in shared memory
// (K rows padded by one word so that 32 lanes reading 32 different rows hit 32 banks),
// then every warp updates its rows: lane j scores key j of the tile, the warp keeps an
// online softmax and accumulates p_j v_j with lanes split over D.  A warp owns
// kRowsPerWarp rows: 4 where there are many rows (fewer K/V tile loads per row), 1 for
// small problems, which are latency-bound and need the CTAs spread over the device.
constexpr int kSimtWarpsT = 8;
constexpr int kKeyTile = 32;
constexpr long long kSimtFewRows = 4096;  // up to this many query rows: one row per warp

template <typename T, int kDPL, int kRowsPerWarp>  // kDPL = D / 32 output dims per lane
__global__ void __launch_bounds__(kSimtWarpsT * 32) attn_simt_kernel(const T* __restrict__ q,
                                                                    const T* __restrict__ k,
                                                                    const T* __restrict__ v, T* __restrict__ out,
                                                                    const int32_t* __restrict__ parent, int B,
                                                                    int Hq, int Hkv, int D, int P, int N, int S,
                                                                    float scale, int32_t* dev_status) {
  constexpr int kD = kDPL * 32;
  constexpr int kRowsCta = kSimtWarpsT * kRowsPerWarp;
  extern __shared__ float simt_smem[];
  // dynamic layout: K tile (rows padded by one word), V tile, the rows' queries, their
  // visible-tree-node masks, the parent array
  float(*s_k)[kD + 1] = reinterpret_cast<float(*)[kD + 1]>(simt_smem);
  float(*s_v)[kD] = reinterpret_cast<float(*)[kD]>(simt_smem + kKeyTile * (kD + 1));
  float(*s_q)[kD] = reinterpret_cast<float(*)[kD]>(simt_smem + kKeyTile * (kD + 1) + kKeyTile * kD);
  uint32_t(*s_vis)[kMaxNodes / 32] = reinterpret_cast<uint32_t(*)[kMaxNodes / 32]>(
      simt_smem + kKeyTile * (kD + 1) + kKeyTile * kD + kRowsCta * kD);
  int* s_par = reinterpret_cast<int*>(simt_smem + kKeyTile * (kD + 1) + kKeyTile * kD + kRowsCta * kD +
                                      kRowsCta * (kMaxNodes / 32));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = Hq / Hkv;
  const int blocks_per_head = (G * N + kRowsCta - 1) / kRowsCta;
  const int kh = (blockIdx.x / blocks_per_head) % Hkv;
  const int b = blockIdx.x / (blocks_per_head * Hkv);
  const int r0 = (blockIdx.x % blocks_per_head) * kRowsCta;
  const int W = (N + 31) / 32;
  const int32_t* par = parent + (size_t)b * N;
  for (int c = threadIdx.x; c < N; c += blockDim.x) s_par[c] = par[c];
  __syncthreads();
  // rows of this CTA: query, visible-node mask (validated ancestor walk)
  for (int rr = warp; rr < kRowsCta; rr += kSimtWarpsT) {
    const int row = r0 + rr;
    const bool live = row < G * N;
    const int g = live ? row / N : 0, i = live ? row % N : 0;
    const size_t qoff = (((size_t)b * Hq + kh * G + g) * N + i) * D;
    for (int d = lane; d < kD; d += 32) s_q[rr][d] = live ? ldx(q, qoff + d) * scale : 0.f;
    for (int w = lane; w < W; w += 32) s_vis[rr][w] = 0u;
    __syncwarp();
    // a padding row of a ragged batch (parent -1 after the last node) has no output;
    // an active row must not follow a padding row
    const bool pad = live && i > 0 && s_par[i] == -1;
    if (lane == 0 && live && !pad) {
      int a = i, guard = 0;
      bool ok = !(i >= 2 && s_par[i - 1] == -1);
      while (a >= 0 && guard <= N) {
        s_vis[rr][a >> 5] |= 1u << (a & 31);
        const int pa = s_par[a];
        if (!(pa < a) || (a == 0 && pa != -1) || (a > 0 && pa < 0)) {
          ok = false;
          break;
        }
        a = pa;
        ++guard;
      }
      if (!ok) {
        set_dev_status(dev_status, TV_DEV_BAD_TREE);
        for (int w = 0; w < W; ++w) s_vis[rr][w] = 0u;
        s_vis[rr][i >> 5] = 1u << (i & 31);
      }
    }
  }
  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kDPL];
#pragma unroll
  for (int rw = 0; rw < kRowsPerWarp; ++rw) {
    m[rw] = -INFINITY;
    l[rw] = 0.f;
#pragma unroll
    for (int t = 0; t < kDPL; ++t) acc[rw][t] = 0.f;
  }
  const size_t kvbase = ((size_t)b * Hkv + kh) * (size_t)S * D;
  const int total = P + N;
  // K/V tiles go through registers: the next tile's loads are issued before the current
  // tile is computed on, so their latency overlaps the compute
  constexpr int kPer = kKeyTile * kD / (kSimtWarpsT * 32);
  float kx[kPer], vx[kPer];
  auto load_tile = [&](int j0) {
#pragma unroll
    for (int it = 0; it < kPer; ++it) {
      const int e = threadIdx.x + it * kSimtWarpsT * 32;
      const int jj = e / kD, d = e - jj * kD;
      const bool in = j0 + jj < total;
      const size_t off = kvbase + (size_t)(j0 + jj) * D + d;
      kx[it] = in ? ldx(k, off) : 0.f;
      vx[it] = in ? ldx(v, off) : 0.f;
    }
  };
  load_tile(0);
  for (int j0 = 0; j0 < total; j0 += kKeyTile) {
    __syncthreads();  // the previous tile is consumed
#pragma unroll
    for (int it = 0; it < kPer; ++it) {
      const int e = threadIdx.x + it * kSimtWarpsT * 32;
      const int jj = e / kD, d = e - jj * kD;
      s_k[jj][d] = kx[it];
      s_v[jj][d] = vx[it];
    }
    __syncthreads();
    if (j0 + kKeyTile < total) load_tile(j0 + kKeyTile);
    const int j = j0 + lane;
#pragma unroll
    for (int rw = 0; rw < kRowsPerWarp; ++rw) {
      const int rr = warp + rw * kSimtWarpsT;
      const int row = r0 + rr;
      if (row >= G * N) continue;  // warp-uniform
      bool vis = j < P;
      if (j >= P && j < total) {
        const int t = j - P;
        vis = (s_vis[rr][t >> 5] >> (t & 31)) & 1u;
      }
      float dot[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
      for (int d = 0; d < kD; d += 4) {
        dot[0] = fmaf(s_q[rr][d], s_k[lane][d], dot[0]);
        dot[1] = fmaf(s_q[rr][d + 1], s_k[lane][d + 1], dot[1]);
        dot[2] = fmaf(s_q[rr][d + 2], s_k[lane][d + 2], dot[2]);
        dot[3] = fmaf(s_q[rr][d + 3], s_k[lane][d + 3], dot[3]);
      }
      const float sc = vis ? (dot[0] + dot[1]) + (dot[2] + dot[3]) : -INFINITY;
      const float mt = warp_max(sc);
      if (mt == -INFINITY) continue;  // nothing visible in this tile for this row
      const float mnew = fmaxf(m[rw], mt);
      const float corr = exp2f((m[rw] - mnew) * kLog2e);
      const float pj = vis ? exp2f((sc - mnew) * kLog2e) : 0.f;
      l[rw] = l[rw] * corr + warp_sum(pj);
#pragma unroll
      for (int t = 0; t < kDPL; ++t) acc[rw][t] *= corr;
#pragma unroll 4
      for (int jj = 0; jj < kKeyTile; ++jj) {
        const float pv = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
        for (int t = 0; t < kDPL; ++t) acc[rw][t] = fmaf(pv, s_v[jj][lane + 32 * t], acc[rw][t]);
      }
      m[rw] = mnew;
    }
  }
#pragma unroll
  for (int rw = 0; rw < kRowsPerWarp; ++rw) {
    const int rr = warp + rw * kSimtWarpsT;
    const int row = r0 + rr;
    if (row >= G * N) continue;
    const int g = row / N, i = row % N;
    if (i > 0 && s_par[i] == -1) continue;  // padding row: nothing written
    const size_t ooff = (((size_t)b * Hq + kh * G + g) * N + i) * D;
    const float inv = l[rw] > 0.f ? 1.f / l[rw] : 0.f;
#pragma unroll
    for (int t = 0; t < kDPL; ++t) stx(out, ooff + lane + 32 * t, acc[rw][t] * inv);
  }
}

static size_t simt_smem_bytes(int d, int rows_cta) {
  return sizeof(float) * ((size_t)kKeyTile * (d + 1) + (size_t)kKeyTile * d + (size_t)rows_cta * d +
                          (size_t)rows_cta * (kMaxNodes / 32) + kMaxNodes);
}

template <typename T, int kRPW>
static void launch_simt_t(const void* q, const void* k, const void* v, void* out, const int32_t* parent, int B,
                          int Hq, int Hkv, int D, int P, int N, int S, float scale, int32_t* dev_status,
                          cudaStream_t stream) {
  constexpr int kRowsCta = kSimtWarpsT * kRPW;
  const int G = Hq / Hkv;
  const long long blocks_per_head = ((long long)G * N + kRowsCta - 1) / kRowsCta;
  const unsigned grid = (unsigned)(blocks_per_head * Hkv * B);
  const T* qq = reinterpret_cast<const T*>(q);
  const T* kk = reinterpret_cast<const T*>(k);
  const T* vv = reinterpret_cast<const T*>(v);
  T* oo = reinterpret_cast<T*>(out);
  switch (D / 32) {
#define TV_SIMT_CASE(n)                                                                                        \
  case n: {                                                                                                    \
    const size_t smem = simt_smem_bytes(n * 32, kRowsCta);                                                     \
    if (cudaFuncSetAttribute(attn_simt_kernel<T, n, kRPW>, cudaFuncAttributeMaxDynamicSharedMemorySize,         \
                             (int)smem) != cudaSuccess)                                                        \
      return;                                                                                                  \
    attn_simt_kernel<T, n, kRPW><<<grid, kSimtWarpsT * 32, smem, stream>>>(qq, kk, vv, oo, parent, B, Hq, Hkv, D, \
                                                                          P, N, S, scale, dev_status);         \
    break;                                                                                                     \
  }
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
  const bool few = (long long)B * Hq * N <= kSimtFewRows;
  if (dtype == TV_BF16) {
    if (few)
      launch_simt_t<uint16_t, 1>(q, k, v, out, parent, B, Hq, Hkv, D, P, N, S, scale, dev_status, stream);
    else
      launch_simt_t<uint16_t, 4>(q, k, v, out, parent, B, Hq, Hkv, D, P, N, S, scale, dev_status, stream);
  } else {
    if (few)
      launch_simt_t<float, 1>(q, k, v, out, parent, B, Hq, Hkv, D, P, N, S, scale, dev_status, stream);
    else
      launch_simt_t<float, 4>(q, k, v, out, parent, B, Hq, Hkv, D, P, N, S, scale, dev_status, stream);
  }
  return cudaGetLastError();
}

}  // namespace tv
