// Tree structure: depth / position ids, ancestor bitmask and child lists.
//
// PTD (Progressive Tree Drafting) §3.1 "tree construction": node v may attend only to
// its observable prefix set pi(v) = {v} U pi(P(v)); its position encoding is fixed by
// |pi(v)|.  One CTA of 1024 threads per sequence; parent[] lives in shared memory.
// Ragged batches: rows after a sequence's last node hold parent -1 (trailing padding);
// they get depth and position -1, an all-zero mask row and no place in the child lists.
#include "philox.cuh"
#include "tv_kernels.cuh"
#include "tv_ptx.cuh"

namespace tv {

__global__ void __launch_bounds__(1024) tree_prep_kernel(const int32_t* __restrict__ parent, int N, int P,
                                                         int32_t* depth, int32_t* pos, uint32_t* anc_mask,
                                                         int32_t* child_off, int32_t* child_idx,
                                                         int32_t* dev_status) {
  __shared__ int s_par[kMaxNodes];
  __shared__ int s_cnt[kMaxNodes + 1];
  __shared__ int s_wsum[32];
  __shared__ int s_bad, s_nact;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int W = (N + 31) / 32;
  if (tid == 0) {
    s_bad = 0;
    s_nact = N;
  }
  __syncthreads();
  for (int i = tid; i < N; i += blockDim.x) {
    const int p = parent[(size_t)b * N + i];
    s_par[i] = p;
    s_cnt[i] = 0;
    if (i >= 1 && p == -1) atomicMin(&s_nact, i);  // the first padding row
  }
  __syncthreads();
  const int n = s_nact;  // active rows 0..n-1
  for (int i = tid; i < N; i += blockDim.x) {
    const int p = s_par[i];
    const bool ok = (i == 0) ? (p == -1) : (i < n ? (p >= 0 && p < i) : (p == -1));
    if (!ok) atomicOr(&s_bad, TV_DEV_BAD_TREE);
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) set_dev_status(dev_status, s_bad);
    return;
  }
  for (int i = tid; i < N; i += blockDim.x) {
    uint32_t* row = anc_mask ? anc_mask + ((size_t)b * N + i) * W : nullptr;
    if (i >= n) {  // padding row
      if (row)
        for (int w = 0; w < W; ++w) row[w] = 0u;
      if (depth) depth[(size_t)b * N + i] = -1;
      if (pos) pos[(size_t)b * N + i] = -1;
      continue;
    }
    // walk i, parent(i), ..., root: indices strictly decrease, so words are visited
    // from high to low and each mask word is written exactly once
    int a = i, d = -1, cw = W - 1;
    uint32_t bits = 0;
    while (a >= 0) {
      const int w = a >> 5;
      while (cw > w) {
        if (row) row[cw] = bits;
        bits = 0;
        --cw;
      }
      bits |= 1u << (a & 31);
      a = s_par[a];
      ++d;
    }
    while (cw >= 0) {
      if (row) row[cw] = bits;
      bits = 0;
      --cw;
    }
    if (depth) depth[(size_t)b * N + i] = d;
    if (pos) pos[(size_t)b * N + i] = P + d;
    if (i > 0) atomicAdd(&s_cnt[s_par[i]], 1);
  }
  if (!child_off) return;
  __syncthreads();
  // exclusive scan of child counts (N <= 1024 = one element per thread)
  const int x = tid < N ? s_cnt[tid] : 0;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_wsum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int v = s_wsum[lane];
    int vi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, vi, o);
      if (lane >= o) vi += y;
    }
    s_wsum[lane] = vi - v;
  }
  __syncthreads();
  const int excl = s_wsum[wid] + incl - x;
  __syncthreads();
  if (tid < N) {
    s_cnt[tid] = excl;
    child_off[(size_t)b * (N + 1) + tid] = excl;
  }
  if (tid == 0) child_off[(size_t)b * (N + 1) + N] = n - 1;
  __syncthreads();
  for (int c = tid + 1; c < n; c += blockDim.x) {
    const int u = s_par[c];
    int rank = 0;
    for (int j = u + 1; j < c; ++j) rank += (s_par[j] == u);
    child_idx[(size_t)b * N + s_cnt[u] + rank] = c;
  }
  // n active nodes have n - 1 edges: the list fills slots 0..n-2, the rest hold -1
  for (int j = n - 1 + tid; j < N; j += blockDim.x) child_idx[(size_t)b * N + j] = -1;
}

cudaError_t launch_tree_prep(const int32_t* parent, int B, int N, int P, int32_t* depth, int32_t* pos,
                             uint32_t* anc_mask, int32_t* child_off, int32_t* child_idx,
                             int32_t* dev_status, cudaStream_t stream) {
  tree_prep_kernel<<<B, 1024, 0, stream>>>(parent, N, P, depth, pos, anc_mask, child_off, child_idx, dev_status);
  return cudaGetLastError();
}

// Self-test of the bounded waits: one warp waits on an mbarrier that nothing arrives on,
// through the same bounded wait every pipeline uses but with the caller's limit; it must
// give up, report TV_DEV_TIMEOUT and return.  (Every other lane of the warp waits on the
// abort flag the first one sets.)
__global__ void wait_selftest_kernel(uint64_t limit_ns, int32_t* dev_status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const bool ok = ptx::mbar_wait_limit(&bar, 0, &abort_flag, limit_ns);
  __syncthreads();
  if (threadIdx.x == 0 && (!ok || abort_flag)) set_dev_status(dev_status, TV_DEV_TIMEOUT);
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, int32_t* dev_status, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, dev_status);
  return cudaGetLastError();
}

// Philox4x32-10 words of caller-given counters under one 64-bit key: the generator the
// sampling walk draws its uniforms from, exposed so that draws can be reproduced.
__global__ void philox_words_kernel(uint64_t seed, const uint32_t* __restrict__ ctr, int n, uint32_t* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint4 c = reinterpret_cast<const uint4*>(ctr)[i];
  const Philox4 r = philox4x32_10(c.x, c.y, c.z, c.w, (uint32_t)seed, (uint32_t)(seed >> 32));
  reinterpret_cast<uint4*>(out)[i] = make_uint4(r.x[0], r.x[1], r.x[2], r.x[3]);
}

cudaError_t launch_philox_words(uint64_t seed, const uint32_t* ctr, int n, uint32_t* out, cudaStream_t stream) {
  if (n > 0) philox_words_kernel<<<(n + 255) / 256, 256, 0, stream>>>(seed, ctr, n, out);
  return cudaGetLastError();
}

}  // namespace tv
