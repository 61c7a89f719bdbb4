// Commit the accepted root path's keys and values into contiguous cache rows.
//
// Speculative-decoding blog, "KV cache handling": the cache entries written for the
// drafted candidates are kept for accepted tokens only.  With the tree's rows at P + t
// (root at P), accepted nodes a_1 < ... < a_L of sequence b move to rows P + 1 .. P + L.
// Since a_k >= k, copying in increasing k never reads a row that an earlier copy of the
// same column wrote; each thread owns one 16-byte column chunk of one (b, kv head, K or V)
// plane, loads all its sources first and then stores, so there is no cross-thread hazard.
#include "tv_kernels.cuh"

namespace tv {

constexpr int kCommitThreads = 256;
constexpr int kCommitBatch = 8;  // rows whose loads are in flight together

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(unsigned char* k_cache, unsigned char* v_cache,
                                                                   const int32_t* accepted,
                                                                   const int32_t* accept_len, int B, int Hkv,
                                                                   int P, int N, long long row_bytes,
                                                                   long long plane_bytes, int chunks,
                                                                   int32_t* dev_status) {
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)B * Hkv * 2 * chunks;
  if (gid >= total) return;
  const int chunk = (int)(gid % chunks);
  const long long plane = gid / chunks;  // (b, h, kv) with kv fastest
  const int kv = (int)(plane & 1);
  const long long bh = plane >> 1;
  const int b = (int)(bh / Hkv);
  const int len = accept_len[b];
  const int32_t* acc = accepted + (size_t)b * N;
  if (len < 0 || len >= N) {
    if (chunk == 0 && plane == (long long)b * Hkv * 2) set_dev_status(dev_status, TV_DEV_BAD_TREE);
    return;
  }
  unsigned char* base = (kv ? v_cache : k_cache) + bh * plane_bytes + (long long)P * row_bytes + chunk * 16;
  int prev = 0;
  for (int k0 = 1; k0 <= len; k0 += kCommitBatch) {
    uint4 val[kCommitBatch];
    bool ok = true;
#pragma unroll
    for (int u = 0; u < kCommitBatch; ++u) {
      const int k = k0 + u;
      if (k <= len) {
        const int a = acc[k - 1];
        ok = ok && a > prev && a < N;  // a root path has increasing node ids
        prev = a;
        val[u] = ok ? *reinterpret_cast<const uint4*>(base + (long long)a * row_bytes) : make_uint4(0, 0, 0, 0);
      }
    }
    if (!ok) {
      if (chunk == 0 && kv == 0) set_dev_status(dev_status, TV_DEV_BAD_TREE);
      return;
    }
#pragma unroll
    for (int u = 0; u < kCommitBatch; ++u) {
      const int k = k0 + u;
      if (k <= len) *reinterpret_cast<uint4*>(base + (long long)k * row_bytes) = val[u];
    }
  }
}

cudaError_t launch_kv_commit(void* k_cache, void* v_cache, const int32_t* accepted, const int32_t* accept_len,
                             int B, int Hkv, int D, int P, int N, int S, tv_dtype dtype, int32_t* dev_status,
                             cudaStream_t stream) {
  const long long elt = dtype == TV_BF16 ? 2 : 4;
  const long long row_bytes = (long long)D * elt;
  const int chunks = (int)(row_bytes / 16);
  const long long total = (long long)B * Hkv * 2 * chunks;
  const unsigned grid = (unsigned)((total + kCommitThreads - 1) / kCommitThreads);
  kv_commit_kernel<<<grid, kCommitThreads, 0, stream>>>(reinterpret_cast<unsigned char*>(k_cache),
                                                         reinterpret_cast<unsigned char*>(v_cache), accepted,
                                                         accept_len, B, Hkv, P, N, row_bytes, (long long)S * row_bytes,
                                                         chunks, dev_status);
  return cudaGetLastError();
}

}  // namespace tv
