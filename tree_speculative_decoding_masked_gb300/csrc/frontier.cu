// One single-drafter tree-expansion step: frontier choice and child attachment.
//
// TreeGraft §3.1: the drafter ranks its candidate pool C_k by the cumulative path score
// s(v) and expands F_k = Top_W(C_k, s); each frontier node's next-token distribution
// contributes its top-m tokens as children with edge score p(u) (the drafter's
// probability) and path score s(child) = s(parent) * p(u).
//
// frontier_topw_kernel: one CTA per sequence ranks the (at most a few thousand) candidate
//   scores by direct comparison (s desc, position asc) and keeps the first W.
// expand_kernel: the drafter rows [R][V] are split over CTAs; each CTA streams its
//   slice once (16-byte loads, several in flight per thread) keeping a running
//   (max, sum 2^(x*c - max)) and a per-thread top-kM list in registers (insertion only
//   when a value beats the list's last entry: rare after the first elements).  Lists are
//   merged warp by warp (kM rounds of a warp arg-max over the lists' heads), the slice's
//   top-m and (max, sum) go to the workspace, and the CTA that completes a row (one
//   acquire-release atomic) merges the row's slices and writes tokens, p and s.
#include <algorithm>

#include "tv_kernels.cuh"
#include "tv_ptx.cuh"

namespace tv {

template <typename T>
__device__ __forceinline__ float to_f32_any(T v);
template <>
__device__ __forceinline__ float to_f32_any<uint16_t>(uint16_t v) {
  return bf16_to_f32(v);
}
template <>
__device__ __forceinline__ float to_f32_any<float>(float v) {
  return v;
}

constexpr int kTopwThreads = 256;
constexpr int kTopwMaxCand = 4096;
constexpr int kExpThreads = 256;
constexpr int kExpMaxSplits = 32;

// ------------------------------------------------------------------------------------
// frontier

__global__ void __launch_bounds__(kTopwThreads) frontier_topw_kernel(const float* scores, const int32_t* count,
                                                                    int C, int W, int32_t* out_idx,
                                                                    int32_t* dev_status) {
  __shared__ float s_sc[kTopwMaxCand];
  const int b = blockIdx.x, t = threadIdx.x;
  int n = count[b];
  if (n < 0 || n > C) {
    if (t == 0) set_dev_status(dev_status, TV_DEV_BAD_TREE);
    n = n < 0 ? 0 : C;
  }
  for (int i = t; i < n; i += blockDim.x) s_sc[i] = scores[(size_t)b * C + i];
  for (int i = t; i < W; i += blockDim.x) out_idx[(size_t)b * W + i] = -1;
  __syncthreads();
  for (int i = t; i < n; i += blockDim.x) {
    const float x = s_sc[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const float y = s_sc[j];
      rank += (y > x) || (y == x && j < i);
    }
    if (rank < W) out_idx[(size_t)b * W + rank] = i;
  }
}

// ------------------------------------------------------------------------------------
// children

struct ExpArgs {
  const void* logits;
  const float* parent_score;
  int R, V, m, S;       // rows, vocabulary, children per row, slices per row
  int chunk;            // elements per slice (a multiple of 8)
  float c2;             // log2(e) / T
  float* part_v;        // [R][S][kM] raw logits of the slice's top list
  int* part_i;          // [R][S][kM] their tokens
  float2* part_ms;      // [R][S] (scaled max, sum)
  unsigned* row_cnt;    // [R]
  int32_t* child_token; // [R][m]
  float* child_p;
  float* child_score;
  int32_t* dev_status;
};

// insert (x, i) into the descending list (v, id) of length kM if it beats the last entry;
// equal values keep the earlier entry in front
template <int kM>
__device__ __forceinline__ void list_insert(float (&v)[kM], int (&id)[kM], float x, int i) {
  if (!(x > v[kM - 1])) return;
#pragma unroll
  for (int k = kM - 1; k >= 0; --k) {
    if (k > 0 && v[k - 1] < x) {
      v[k] = v[k - 1];
      id[k] = id[k - 1];
    } else if (v[k] < x) {
      v[k] = x;
      id[k] = i;
    }
  }
}

// kM rounds of a warp arg-max over the lanes' list heads (value desc, token asc); round r's
// winner lands in out_v[r], out_i[r] (written by lane 0)
template <int kM>
__device__ __forceinline__ void warp_merge_lists(float (&v)[kM], int (&id)[kM], float* out_v, int* out_i) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int r = 0; r < kM; ++r) {
    float bv = v[0];
    int bi = id[0], bl = lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const int ol = __shfl_xor_sync(0xffffffffu, bl, o);
      if (ov > bv || (ov == bv && (oi < bi || (oi == bi && ol < bl)))) {
        bv = ov;
        bi = oi;
        bl = ol;
      }
    }
    if (lane == 0) {
      out_v[r] = bv;
      out_i[r] = bi;
    }
    if (lane == bl) {  // pop the winner's head
#pragma unroll
      for (int k = 0; k + 1 < kM; ++k) {
        v[k] = v[k + 1];
        id[k] = id[k + 1];
      }
      v[kM - 1] = -INFINITY;
      id[kM - 1] = 0x7fffffff;
    }
  }
}

template <typename T>
__device__ __forceinline__ void unpack8(const uint4& u, float* x);
template <>
__device__ __forceinline__ void unpack8<uint16_t>(const uint4& u, float* x) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(w[k] << 16);
    x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}
template <>
__device__ __forceinline__ void unpack8<float>(const uint4& u, float* x) {
  x[0] = __uint_as_float(u.x);
  x[1] = __uint_as_float(u.y);
  x[2] = __uint_as_float(u.z);
  x[3] = __uint_as_float(u.w);
}

template <typename T, int kM, bool kVec>
__global__ void __launch_bounds__(kExpThreads) expand_kernel(ExpArgs a) {
  __shared__ float s_v[kExpThreads / 32][kM];
  __shared__ int s_i[kExpThreads / 32][kM];
  __shared__ float2 s_ms[kExpThreads / 32];
  __shared__ float s_fv[kM];
  __shared__ int s_fi[kM];
  __shared__ int s_last;
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int row = blockIdx.x / a.S, slice = blockIdx.x % a.S;
  const int v0 = min(a.V, slice * a.chunk), v1 = min(a.V, v0 + a.chunk);
  const T* x = reinterpret_cast<const T*>(a.logits) + (size_t)row * a.V;
  float lv[kM];
  int li[kM];
#pragma unroll
  for (int k = 0; k < kM; ++k) {
    lv[k] = -INFINITY;
    li[k] = 0x7fffffff;
  }
  float mc = -INFINITY, sum = 0.f;
  auto push = [&](float xv, int i) {
    if (xv * a.c2 > mc) {
      const float nm = xv * a.c2;
      sum *= ptx::ex2(mc - nm);
      mc = nm;
    }
    sum += ptx::ex2(fmaf(xv, a.c2, -mc));
    list_insert<kM>(lv, li, xv, i);
  };
  if constexpr (kVec) {
    constexpr int kN = 16 / sizeof(T);
    const uint4* p = reinterpret_cast<const uint4*>(x + v0);
    const int nvec = (v1 - v0) / kN;
    constexpr int kB = 4;  // 16-byte loads in flight per thread
    for (int jb = t; jb < nvec; jb += kB * kExpThreads) {
      uint4 u[kB];
#pragma unroll
      for (int q = 0; q < kB; ++q) {
        const int j = jb + q * kExpThreads;
        u[q] = j < nvec ? __ldcs(p + j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < kB; ++q) {
        const int j = jb + q * kExpThreads;
        if (j < nvec) {
          float xv[kN];
          unpack8<T>(u[q], xv);
          // whole-vector fast path: one max, one rare rescale, a tree of exponentials,
          // and the list touched only if the vector's max beats its last entry
          float vm = xv[0];
#pragma unroll
          for (int e = 1; e < kN; ++e) vm = fmaxf(vm, xv[e]);
          if (vm * a.c2 > mc) {
            const float nm = vm * a.c2;
            sum *= ptx::ex2(mc - nm);
            mc = nm;
          }
          float ex[kN];
#pragma unroll
          for (int e = 0; e < kN; ++e) ex[e] = ptx::ex2(fmaf(xv[e], a.c2, -mc));
#pragma unroll
          for (int w = 1; w < kN; w *= 2)
#pragma unroll
            for (int e = 0; e + w < kN; e += 2 * w) ex[e] += ex[e + w];
          sum += ex[0];
          if (vm > lv[kM - 1]) {
#pragma unroll
            for (int e = 0; e < kN; ++e) list_insert<kM>(lv, li, xv[e], v0 + j * kN + e);
          }
        }
      }
    }
    for (int i = v0 + nvec * kN + t; i < v1; i += kExpThreads) push(to_f32_any<T>(x[i]), i);
  } else {
    for (int i = v0 + t; i < v1; i += kExpThreads) push(to_f32_any<T>(x[i]), i);
  }
  // slice (max, sum): warp then CTA
  float wm = mc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
  float ws = sum > 0.f ? sum * ptx::ex2(mc - wm) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
  if (lane == 0) s_ms[wid] = make_float2(wm, ws);
  // slice top list: per warp, then across warps
  warp_merge_lists<kM>(lv, li, s_v[wid], s_i[wid]);
  __syncthreads();
  const size_t slot = (size_t)row * a.S + slice;
  if (wid == 0) {
    float cm = lane < kExpThreads / 32 ? s_ms[lane].x : -INFINITY;
    float cmax = cm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
    float cs = (lane < kExpThreads / 32 && s_ms[lane].y > 0.f) ? s_ms[lane].y * ptx::ex2(cm - cmax) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, o);
#pragma unroll
    for (int k = 0; k < kM; ++k) {
      lv[k] = lane < kExpThreads / 32 ? s_v[lane][k] : -INFINITY;
      li[k] = lane < kExpThreads / 32 ? s_i[lane][k] : 0x7fffffff;
    }
    warp_merge_lists<kM>(lv, li, s_fv, s_fi);
    __syncwarp();
    for (int k = lane; k < kM; k += 32) {
      a.part_v[slot * kM + k] = s_fv[k];
      a.part_i[slot * kM + k] = s_fi[k];
    }
    if (lane == 0) a.part_ms[slot] = make_float2(cmax, cs);
  }
  // the CTA that completes the row merges its slices
  __syncthreads();
  if (t == 0) {
    const unsigned prev = ptx::atom_add_acq_rel_gpu(a.row_cnt + row, 1u);
    s_last = prev + 1 == (unsigned)a.S;
    if (s_last) a.row_cnt[row] = 0;
  }
  __syncthreads();
  if (!s_last || wid != 0) return;
  const size_t base = (size_t)row * a.S;
  float2 ms = lane < a.S ? __ldcg(a.part_ms + base + lane) : make_float2(-INFINITY, 0.f);
  float rmax = ms.x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, o));
  float rs = ms.y > 0.f ? ms.y * ptx::ex2(ms.x - rmax) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
  const float lse2 = rmax + log2f(rs);
#pragma unroll
  for (int k = 0; k < kM; ++k) {
    lv[k] = lane < a.S ? __ldcg(a.part_v + (base + lane) * kM + k) : -INFINITY;
    li[k] = lane < a.S ? __ldcg(a.part_i + (base + lane) * kM + k) : 0x7fffffff;
  }
  warp_merge_lists<kM>(lv, li, s_fv, s_fi);
  __syncwarp();
  const float ps = a.parent_score[row];
  for (int k = lane; k < a.m; k += 32) {
    const bool ok = k < a.V;
    const float p = ok ? ptx::ex2(fmaf(s_fv[k], a.c2, -lse2)) : 0.f;
    a.child_token[(size_t)row * a.m + k] = ok ? s_fi[k] : -1;
    a.child_p[(size_t)row * a.m + k] = p;
    a.child_score[(size_t)row * a.m + k] = ok ? __fmul_rn(ps, p) : 0.f;
  }
}

// ------------------------------------------------------------------------------------
// host side

static int exp_km(int m) { return m <= 4 ? 4 : m <= 8 ? 8 : m <= 16 ? 16 : 32; }

static void exp_plan(int R, int V, int& S, int& chunk) {
  // about two CTAs per SM of the 152 (the per-slice merges are not free), at least 4096
  // elements per slice
  const long long want = (2LL * 152 + R - 1) / R;
  S = (int)std::min<long long>(std::max<long long>(1, want), kExpMaxSplits);
  S = std::min(S, std::max(1, V / 4096));
  chunk = (V + S - 1) / S;
  chunk = (chunk + 7) / 8 * 8;
  S = (V + chunk - 1) / chunk;
}

size_t expand_ws_bytes(int R, int V, int m) {
  if (R < 1 || V < 1 || m < 1) return 0;
  int S, chunk;
  exp_plan(R, V, S, chunk);
  const size_t km = exp_km(m);
  size_t off = 0;
  off += (size_t)R * S * km * 4;  // part_v
  off += (size_t)R * S * km * 4;  // part_i
  off = (off + 15) / 16 * 16;
  off += (size_t)R * S * 8;  // part_ms
  off += (size_t)R * 4;      // row_cnt
  return (off + 255) / 256 * 256;
}

cudaError_t launch_frontier_topw(const float* scores, const int32_t* count, int B, int C, int W, int32_t* out_idx,
                                 int32_t* dev_status, cudaStream_t stream) {
  frontier_topw_kernel<<<B, kTopwThreads, 0, stream>>>(scores, count, C, W, out_idx, dev_status);
  return cudaGetLastError();
}

template <typename T, int kM>
static cudaError_t launch_expand_t(const ExpArgs& a, bool vec, cudaStream_t stream) {
  const unsigned grid = (unsigned)((long long)a.R * a.S);
  if (vec)
    expand_kernel<T, kM, true><<<grid, kExpThreads, 0, stream>>>(a);
  else
    expand_kernel<T, kM, false><<<grid, kExpThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_expand_m(const ExpArgs& a, bool vec, cudaStream_t stream) {
  switch (exp_km(a.m)) {
    case 4:
      return launch_expand_t<T, 4>(a, vec, stream);
    case 8:
      return launch_expand_t<T, 8>(a, vec, stream);
    case 16:
      return launch_expand_t<T, 16>(a, vec, stream);
    default:
      return launch_expand_t<T, 32>(a, vec, stream);
  }
}

cudaError_t launch_expand(const void* logits, const float* parent_score, int R, int V, int m, float temperature,
                          tv_dtype dtype, int32_t* child_token, float* child_p, float* child_score, char* ws,
                          int32_t* dev_status, cudaStream_t stream) {
  ExpArgs a;
  a.logits = logits;
  a.parent_score = parent_score;
  a.R = R;
  a.V = V;
  a.m = m;
  exp_plan(R, V, a.S, a.chunk);
  a.c2 = kLog2e / temperature;
  const size_t km = exp_km(m);
  size_t off = 0;
  a.part_v = reinterpret_cast<float*>(ws + off);
  off += (size_t)R * a.S * km * 4;
  a.part_i = reinterpret_cast<int*>(ws + off);
  off += (size_t)R * a.S * km * 4;
  off = (off + 15) / 16 * 16;
  a.part_ms = reinterpret_cast<float2*>(ws + off);
  off += (size_t)R * a.S * 8;
  a.row_cnt = reinterpret_cast<unsigned*>(ws + off);
  a.child_token = child_token;
  a.child_p = child_p;
  a.child_score = child_score;
  a.dev_status = dev_status;
  const size_t esz = dtype == TV_BF16 ? 2 : 4;
  const bool vec = ((size_t)V * esz) % 16 == 0 && (reinterpret_cast<uintptr_t>(logits) % 16) == 0 &&
                   ((size_t)a.chunk * esz) % 16 == 0;
  return dtype == TV_BF16 ? launch_expand_m<uint16_t>(a, vec, stream) : launch_expand_m<float>(a, vec, stream);
}

}  // namespace tv
