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
//   (max, sum 2^(x*c - max)) per thread and a sorted top-m list per warp (lane k holds
//   the k-th best): a vector touches the list only if its max reaches the list's m-th
//   entry, and each qualifying element is inserted by the whole warp (ballot for the
//   position, one shuffle to shift the tail).  Warp 0 merges the warps' lists, the
//   slice's top-m and (max, sum) go to the workspace, and the CTA that completes a row
//   (one acquire-release atomic) merges the row's slices and writes tokens, p and s.
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
  float* part_v;        // [R][S][32] raw logits of the slice's top list
  int* part_i;          // [R][S][32] their tokens
  float2* part_ms;      // [R][S] (scaled max, sum)
  unsigned* row_cnt;    // [R]
  int32_t* child_token; // [R][m]
  float* child_p;
  float* child_score;
  int32_t* dev_status;
};

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

// A warp-wide sorted list of the best (value, token) pairs seen so far: lane k holds the
// k-th best (value descending, token ascending), lanes >= m hold nothing.  An insertion
// is warp-collective: every lane compares its entry with the candidate, the lanes behind
// it shift down by one.
struct WarpList {
  float v;
  int i;
  __device__ __forceinline__ void init() {
    v = -INFINITY;
    i = 0x7fffffff;
  }
  __device__ __forceinline__ static bool better(float xa, int ia, float xb, int ib) {
    return xa > xb || (xa == xb && ia < ib);
  }
  // the m-th best entry (the bar a candidate must beat)
  __device__ __forceinline__ void bar(int m, float& bv, int& bi) const {
    bv = __shfl_sync(0xffffffffu, v, m - 1);
    bi = __shfl_sync(0xffffffffu, i, m - 1);
  }
  // warp-uniform candidate (x, ix)
  __device__ __forceinline__ void insert(float x, int ix, int m) {
    const int lane = threadIdx.x & 31;
    const unsigned ahead = __ballot_sync(0xffffffffu, lane < m && better(v, i, x, ix));
    const int pos = __popc(ahead);
    const float pv = __shfl_up_sync(0xffffffffu, v, 1);
    const int pi = __shfl_up_sync(0xffffffffu, i, 1);
    if (pos < m) {
      if (lane == pos) {
        v = x;
        i = ix;
      } else if (lane > pos && lane < m) {
        v = pv;
        i = pi;
      }
    }
  }
  // merge another sorted list (lane k holds its k-th best) and keep the best 32: the
  // concatenation of this list and the other reversed is bitonic, so one comparison with
  // the mirrored lane keeps the better half and five shuffle stages sort it
  __device__ __forceinline__ void merge(float ov, int oi) {
    const int lane = threadIdx.x & 31;
    const float rv = __shfl_sync(0xffffffffu, ov, 31 - lane);
    const int ri = __shfl_sync(0xffffffffu, oi, 31 - lane);
    if (better(rv, ri, v, i)) {
      v = rv;
      i = ri;
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
      const float pv = __shfl_xor_sync(0xffffffffu, v, d);
      const int pi = __shfl_xor_sync(0xffffffffu, i, d);
      const bool pb = better(pv, pi, v, i);
      if (((lane & d) == 0) == pb) {
        v = pv;
        i = pi;
      }
    }
  }
  // become the sorted list of the lanes' (x, ix): a bitonic sort across the warp
  __device__ __forceinline__ void sort_from(float x, int ix) {
    const int lane = threadIdx.x & 31;
    v = x;
    i = ix;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const float pv = __shfl_xor_sync(0xffffffffu, v, j);
        const int pi = __shfl_xor_sync(0xffffffffu, i, j);
        const bool lower = (lane & j) == 0, desc = (lane & k) == 0;
        const bool pb = better(pv, pi, v, i);
        if ((lower == desc) == pb) {
          v = pv;
          i = pi;
        }
      }
  }
  // offer each lane's (x, ix) (per-lane candidates, in lane order)
  __device__ __forceinline__ void offer(float x, int ix, bool want, int m) {
    float bv;
    int bi;
    bar(m, bv, bi);
    unsigned cand = __ballot_sync(0xffffffffu, want && better(x, ix, bv, bi));
    while (cand) {
      const int src = __ffs(cand) - 1;
      cand &= cand - 1;
      const float cx = __shfl_sync(0xffffffffu, x, src);
      const int ci = __shfl_sync(0xffffffffu, ix, src);
      float b2;
      int i2;
      bar(m, b2, i2);
      if (better(cx, ci, b2, i2)) insert(cx, ci, m);
    }
  }
};

template <typename T, bool kVec>
__global__ void __launch_bounds__(kExpThreads) expand_kernel(ExpArgs a) {
  __shared__ float s_v[kExpThreads / 32][32];
  __shared__ int s_i[kExpThreads / 32][32];
  __shared__ float2 s_ms[kExpThreads / 32];
  __shared__ int s_last;
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int m = a.m;
  const int row = blockIdx.x / a.S, slice = blockIdx.x % a.S;
  const int v0 = min(a.V, slice * a.chunk), v1 = min(a.V, v0 + a.chunk);
  const T* x = reinterpret_cast<const T*>(a.logits) + (size_t)row * a.V;
  WarpList wl;
  wl.init();
  float mc = -INFINITY, sum = 0.f;
  auto scalar = [&](int i, bool ok) {  // one element per lane (tails and unaligned rows)
    const float xv = ok ? to_f32_any<T>(x[i]) : -INFINITY;
    if (ok) {
      if (xv * a.c2 > mc) {
        const float nm = xv * a.c2;
        sum *= ptx::ex2(mc - nm);
        mc = nm;
      }
      sum += ptx::ex2(fmaf(xv, a.c2, -mc));
    }
    wl.offer(xv, i, ok, m);
  };
  if constexpr (kVec) {
    constexpr int kN = 16 / sizeof(T);
    const uint4* p = reinterpret_cast<const uint4*>(x + v0);
    const int nvec = (v1 - v0) / kN;
    constexpr int kB = 4;  // 16-byte loads in flight per thread
    for (int jb = t - lane; jb < nvec; jb += kB * kExpThreads) {  // warp-uniform trip count
      uint4 u[kB];
#pragma unroll
      for (int q = 0; q < kB; ++q) {
        const int j = jb + lane + q * kExpThreads;
        u[q] = j < nvec ? __ldcs(p + j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < kB; ++q) {
        const int j = jb + lane + q * kExpThreads;
        const bool ok = j < nvec;
        float xv[kN];
        unpack8<T>(u[q], xv);
        float vm = -INFINITY;
        int em = 0;  // position of the vector's max (first one on ties)
        if (ok) {
          vm = xv[0];
#pragma unroll
          for (int e = 1; e < kN; ++e)
            if (xv[e] > vm) {
              vm = xv[e];
              em = e;
            }
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
        }
        if (jb == t - lane && q == 0) {
          // first vectors of the warp: the lanes' maxima, sorted, seed the list in one go
          // (real elements, so its m-th entry is a valid bar from the start)
          wl.sort_from(vm, ok ? v0 + j * kN + em : 0x7fffffff);
          if (lane >= m) wl.init();
          float bv;
          int bi;
          wl.bar(m, bv, bi);
#pragma unroll
          for (int e = 0; e < kN; ++e) wl.offer(xv[e], v0 + j * kN + e, ok && e != em && vm >= bv, m);
        } else {
          // the list is touched only by vectors whose max reaches the warp's m-th entry
          float bv;
          int bi;
          wl.bar(m, bv, bi);
          if (__any_sync(0xffffffffu, ok && vm >= bv)) {
#pragma unroll
            for (int e = 0; e < kN; ++e) wl.offer(xv[e], v0 + j * kN + e, ok && vm >= bv, m);
          }
        }
      }
    }
    const int tail0 = v0 + nvec * kN;
    for (int ib = tail0 + t - lane; ib < v1; ib += kExpThreads) scalar(ib + lane, ib + lane < v1);
  } else {
    for (int ib = v0 + t - lane; ib < v1; ib += kExpThreads) scalar(ib + lane, ib + lane < v1);
  }
  // slice (max, sum): warp then CTA; slice list: the warps' lists merged by warp 0
  float wm = mc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
  float ws = sum > 0.f ? sum * ptx::ex2(mc - wm) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
  if (lane == 0) s_ms[wid] = make_float2(wm, ws);
  s_v[wid][lane] = wl.v;
  s_i[wid][lane] = wl.i;
  __syncthreads();
  const size_t slot = (size_t)row * a.S + slice;
  if (wid == 0) {
    const float cm = lane < kExpThreads / 32 ? s_ms[lane].x : -INFINITY;
    float cmax = cm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
    float cs = (lane < kExpThreads / 32 && s_ms[lane].y > 0.f) ? s_ms[lane].y * ptx::ex2(cm - cmax) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, o);
    for (int w2 = 1; w2 < kExpThreads / 32; ++w2) wl.merge(s_v[w2][lane], s_i[w2][lane]);
    if (lane < m) {
      a.part_v[slot * 32 + lane] = wl.v;
      a.part_i[slot * 32 + lane] = wl.i;
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
  if (!s_last) return;
  const size_t base = (size_t)row * a.S;
  // every warp merges a share of the row's slice lists, then warp 0 merges the warps'
  wl.init();
  for (int sl = wid; sl < a.S; sl += kExpThreads / 32) {
    const float pv = lane < m ? __ldcg(a.part_v + (base + sl) * 32 + lane) : -INFINITY;
    const int pi = lane < m ? __ldcg(a.part_i + (base + sl) * 32 + lane) : 0x7fffffff;
    wl.merge(pv, pi);
  }
  s_v[wid][lane] = wl.v;
  s_i[wid][lane] = wl.i;
  __syncthreads();
  if (wid != 0) return;
  for (int w2 = 1; w2 < kExpThreads / 32; ++w2) wl.merge(s_v[w2][lane], s_i[w2][lane]);
  const float2 ms = lane < a.S ? __ldcg(a.part_ms + base + lane) : make_float2(-INFINITY, 0.f);
  float rmax = ms.x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, o));
  float rs = ms.y > 0.f ? ms.y * ptx::ex2(ms.x - rmax) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
  const float lse2 = rmax + log2f(rs);
  const float ps = a.parent_score[row];
  if (lane < m) {
    const bool ok = lane < a.V;
    const float pr = ok ? ptx::ex2(fmaf(wl.v, a.c2, -lse2)) : 0.f;
    a.child_token[(size_t)row * m + lane] = ok ? wl.i : -1;
    a.child_p[(size_t)row * m + lane] = pr;
    a.child_score[(size_t)row * m + lane] = ok ? __fmul_rn(ps, pr) : 0.f;
  }
}

// ------------------------------------------------------------------------------------
// host side

static int exp_km(int) { return 32; }  // slice lists are stored with 32 slots

static void exp_plan(int R, int V, int& S, int& chunk) {
  // about two CTAs per SM of the 152, but at least 16384 elements per slice: every slice
  // pays a list seed, a CTA merge and a share of the row merge
  const long long want = (2LL * 152 + R - 1) / R;
  S = (int)std::min<long long>(std::max<long long>(1, want), kExpMaxSplits);
  S = std::min(S, std::max(1, V / 16384));
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

template <typename T>
static cudaError_t launch_expand_t(const ExpArgs& a, bool vec, cudaStream_t stream) {
  const unsigned grid = (unsigned)((long long)a.R * a.S);
  if (vec)
    expand_kernel<T, true><<<grid, kExpThreads, 0, stream>>>(a);
  else
    expand_kernel<T, false><<<grid, kExpThreads, 0, stream>>>(a);
  return cudaGetLastError();
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
  return dtype == TV_BF16 ? launch_expand_t<uint16_t>(a, vec, stream) : launch_expand_t<float>(a, vec, stream);
}

}  // namespace tv
