// Fused per-node vocabulary pass and greedy acceptance walk.
//
// Speculative-decoding blog, "greedy decoding, intuitive version" / "acceptance
// probability for sampling": every drafted position needs the target's choice (argmax)
// and the target probability of the drafted token p_u(t).  One streaming, vectorised
// read of each logits row yields argmax (lowest index among equal raw values) and the
// base-2 log-sum-exp of x/T; rows are split across CTAs and the last CTA of a row merges
// the partials, the last row of a sequence runs that sequence's epilogue (drafted-token
// probabilities and, for greedy verification, the walk down the tree).
#include "tv_kernels.cuh"
#include "tv_ptx.cuh"

namespace tv {

constexpr int kStagedParts = 640;  // split partials staged in shared memory by the merging CTA

struct VocabPartial {
  float m;   // max of x * c2 over the chunk (base-2 scaled)
  float s;   // sum 2^(x*c2 - m)
  float av;  // raw max value
  int ai;    // its lowest index
};

template <typename T>
struct Vec16;
template <>
struct Vec16<uint16_t> {
  static constexpr int kN = 8;
};
template <>
struct Vec16<float> {
  static constexpr int kN = 4;
};

__device__ __forceinline__ float to_f32(uint16_t x) { return bf16_to_f32(x); }
__device__ __forceinline__ float to_f32(float x) { return x; }

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& u, float* out);
template <>
__device__ __forceinline__ void unpack16<uint16_t>(const uint4& u, float* out) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    out[2 * k] = __uint_as_float(w[k] << 16);
    out[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}
template <>
__device__ __forceinline__ void unpack16<float>(const uint4& u, float* out) {
  out[0] = __uint_as_float(u.x);
  out[1] = __uint_as_float(u.y);
  out[2] = __uint_as_float(u.z);
  out[3] = __uint_as_float(u.w);
}

// Running state of one thread over its share of a row.
struct RowAcc {
  float av;  // raw max
  int ai;
  float mc;  // av * c2 (rounded once)
  float s;
  __device__ __forceinline__ void init() {
    av = -INFINITY;
    ai = 0x7fffffff;
    mc = -INFINITY;
    s = 0.f;
  }
  template <int kN>
  __device__ __forceinline__ void push(const float* x, int base, float c2) {
    float bv = x[0];
    int bi = base;
#pragma unroll
    for (int k = 1; k < kN; ++k)
      if (x[k] > bv) {
        bv = x[k];
        bi = base + k;
      }
    if (bv > av) {
      float nmc = bv * c2;
      s *= ptx::ex2(mc - nmc);
      av = bv;
      ai = bi;
      mc = nmc;
    }
#pragma unroll
    for (int k = 0; k < kN; ++k) s += ptx::ex2(fmaf(x[k], c2, -mc));
  }
  __device__ __forceinline__ void push1(float x, int idx, float c2) {
    if (x > av) {
      float nmc = x * c2;
      s *= ptx::ex2(mc - nmc);
      av = x;
      ai = idx;
      mc = nmc;
    }
    s += ptx::ex2(fmaf(x, c2, -mc));
  }
};

__device__ __forceinline__ VocabPartial partial_merge(VocabPartial a, VocabPartial b) {
  VocabPartial r;
  MaxSum ms = maxsum_merge({a.m, a.s}, {b.m, b.s});
  ArgMax am = argmax_merge({a.av, a.ai}, {b.av, b.ai});
  r.m = ms.m;
  r.s = ms.s;
  r.av = am.v;
  r.ai = am.i;
  return r;
}

__device__ __forceinline__ VocabPartial warp_merge(VocabPartial p) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    VocabPartial q;
    q.m = __shfl_xor_sync(0xffffffffu, p.m, o);
    q.s = __shfl_xor_sync(0xffffffffu, p.s, o);
    q.av = __shfl_xor_sync(0xffffffffu, p.av, o);
    q.ai = __shfl_xor_sync(0xffffffffu, p.ai, o);
    p = partial_merge(p, q);
  }
  return p;
}

// Block-wide merge; result valid in thread 0.  Uses `red` (>= 32 entries).
__device__ __forceinline__ VocabPartial block_merge(VocabPartial p, VocabPartial* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  p = warp_merge(p);
  if (lane == 0) red[wid] = p;
  __syncthreads();
  if (wid == 0) {
    VocabPartial q = lane < nw ? red[lane] : VocabPartial{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
    q = warp_merge(q);
    if (lane == 0) red[0] = q;
  }
  __syncthreads();
  VocabPartial r = red[0];
  __syncthreads();
  return r;
}

// Accumulate x[v0, v1) of one row into `acc`: 16-byte streaming loads, eight in flight
// per thread, when kVec; scalar loads otherwise.
template <typename T, bool kVec>
__device__ __forceinline__ void scan_chunk(const T* __restrict__ row, int v0, int v1, float c2, RowAcc& acc) {
  if constexpr (kVec) {
    constexpr int kN = Vec16<T>::kN;
    constexpr int kInFlight = 8;
    const int nvec = (v1 - v0) / kN;
    const uint4* p = reinterpret_cast<const uint4*>(row + v0);
    const int stride = blockDim.x;
    for (int j = threadIdx.x; j < nvec; j += kInFlight * stride) {
      uint4 u[kInFlight];
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int idx = j + k * stride;
        if (idx < nvec) u[k] = __ldcs(p + idx);
      }
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int idx = j + k * stride;
        if (idx < nvec) {
          float x[kN];
          unpack16<T>(u[k], x);
          acc.template push<kN>(x, v0 + idx * kN, c2);
        }
      }
    }
    for (int v = v0 + nvec * kN + threadIdx.x; v < v1; v += stride) acc.push1(to_f32(row[v]), v, c2);
  } else {
    for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) acc.push1(to_f32(row[v]), v, c2);
  }
}

struct VocabArgs {
  const void* logits;
  const void* draft;  // sampling only
  const int32_t* parent;
  const int32_t* tokens;
  int B, N, V, splits, chunk;
  float c2;  // log2(e) / T
  VocabPartial* part;
  VocabPartial* part_q;
  float* lse2;    // [rows] base-2 lse of x*c2
  float* lse2_q;  // [rows]
  int32_t* amax;  // [rows]
  float* pc;      // [rows] p_{parent(c)}(t_c) (fp32), sampling scratch
  float* qc;
  unsigned* row_cnt;  // [rows]
  unsigned* seq_cnt;  // [B]
  // outputs
  int32_t* accepted;
  int32_t* accept_len;
  int32_t* bonus;
  float* p_draft;
  float* q_draft;
  float* row_lse;
  int32_t* row_argmax;
  int32_t* dev_status;
  int sampling;
};

template <typename T>
__device__ __forceinline__ float load_logit(const void* base, size_t idx) {
  return to_f32(reinterpret_cast<const T*>(base)[idx]);
}

// Per-sequence epilogue, run by the CTA that finished the sequence's last partial.
// s_lse2 / s_lse2q / s_am hold the merged row statistics of sequence b.
template <typename T>
__device__ void sequence_epilogue(const VocabArgs& a, int b, const float* s_lse2, const float* s_lse2q,
                                  const int* s_am) {
  __shared__ int s_par[kMaxNodes];
  __shared__ int s_tok[kMaxNodes];
  __shared__ int s_bad;
  const int N = a.N, V = a.V;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  for (int c = threadIdx.x; c < N; c += blockDim.x) {
    int p = a.parent[(size_t)b * N + c];
    int t = a.tokens[(size_t)b * N + c];
    s_par[c] = p;
    s_tok[c] = t;
    bool ok = (c == 0) ? (p == -1) : (p >= 0 && p < c);
    if (!ok) atomicOr(&s_bad, TV_DEV_BAD_TREE);
    if (c > 0 && (t < 0 || t >= V)) atomicOr(&s_bad, TV_DEV_BAD_TOKEN);
  }
  __syncthreads();
  const int bad = s_bad;
  if (bad && threadIdx.x == 0) set_dev_status(a.dev_status, bad);
  // drafted-token probabilities p_c = 2^(x[parent(c)][t_c] * c2 - lse2[parent(c)])
  for (int c = threadIdx.x; c < N; c += blockDim.x) {
    float pv = __int_as_float(0x7fc00000), qv = pv;
    if (c > 0 && !bad) {
      int u = s_par[c];
      size_t idx = ((size_t)b * N + u) * (size_t)V + s_tok[c];
      pv = ptx::ex2(fmaf(load_logit<T>(a.logits, idx), a.c2, -s_lse2[u]));
      if (a.sampling) qv = ptx::ex2(fmaf(load_logit<T>(a.draft, idx), a.c2, -s_lse2q[u]));
    }
    if (a.pc) a.pc[(size_t)b * N + c] = pv;
    if (a.qc) a.qc[(size_t)b * N + c] = qv;
    if (a.p_draft) a.p_draft[(size_t)b * N + c] = pv;
    if (a.q_draft) a.q_draft[(size_t)b * N + c] = qv;
  }
  if (a.sampling) return;  // the sampling walk runs in its own kernel
  // greedy walk: first find, in parallel, each node's child whose token equals the
  // node's argmax (lowest index if several), then follow those links from the root
  __shared__ int s_match[kMaxNodes];
  __shared__ int s_path[kMaxNodes];
  __shared__ int s_len, s_bonus;
  for (int c = threadIdx.x; c < N; c += blockDim.x) s_match[c] = 0x7fffffff;
  __syncthreads();
  if (!bad)
    for (int c = 1 + threadIdx.x; c < N; c += blockDim.x)
      if (s_tok[c] == s_am[s_par[c]]) atomicMin(&s_match[s_par[c]], c);
  __syncthreads();
  if (threadIdx.x == 0) {
    int cur = 0, len = 0;
    if (!bad) {
      for (int nxt = s_match[0]; nxt != 0x7fffffff; nxt = s_match[cur]) {
        s_path[len++] = nxt;
        cur = nxt;
      }
    }
    s_len = len;
    s_bonus = bad ? -1 : s_am[cur];
  }
  __syncthreads();
  const int len = s_len;
  for (int j = threadIdx.x; j < N; j += blockDim.x) a.accepted[(size_t)b * N + j] = j < len ? s_path[j] : -1;
  if (threadIdx.x == 0) {
    a.accept_len[b] = len;
    a.bonus[b] = s_bonus;
  }
}

template <typename T, bool kVec>
__global__ void __launch_bounds__(256, 4) vocab_pass_kernel(VocabArgs a) {
  __shared__ VocabPartial red[32];
  __shared__ int s_flag;
  __shared__ float s_lse2[kMaxNodes];
  __shared__ float s_lse2q[kMaxNodes];
  __shared__ int s_am[kMaxNodes];
  __shared__ float4 s_stage[kStagedParts];
  const int split = blockIdx.x % a.splits;
  const int row = blockIdx.x / a.splits;
  const int b = row / a.N;
  const int v0 = split * a.chunk;
  const int v1 = min(a.V, v0 + a.chunk);
  const size_t roff = (size_t)row * a.V;

  RowAcc acc;
  acc.init();
  if (v0 < v1) scan_chunk<T, kVec>(reinterpret_cast<const T*>(a.logits) + roff, v0, v1, a.c2, acc);
  VocabPartial p = block_merge({acc.mc, acc.s, acc.av, acc.ai}, red);
  VocabPartial pq{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
  if (a.sampling) {
    RowAcc accq;
    accq.init();
    if (v0 < v1) scan_chunk<T, kVec>(reinterpret_cast<const T*>(a.draft) + roff, v0, v1, a.c2, accq);
    pq = block_merge({accq.mc, accq.s, accq.av, accq.ai}, red);
  }
  if (threadIdx.x == 0) {
    a.part[(size_t)row * a.splits + split] = p;
    if (a.sampling) a.part_q[(size_t)row * a.splits + split] = pq;
    __threadfence();
    // one completion counter per sequence: the CTA that writes its last partial merges
    const unsigned prev = atomicAdd(a.seq_cnt + b, 1u);
    s_flag = (prev == (unsigned)(a.N * a.splits - 1));
  }
  __syncthreads();
  if (!s_flag) return;
  __threadfence();
  // merge the splits of every row of sequence b.  All partials are fetched at once (one
  // round trip), staged in shared memory, then merged per row.
  const int npart = a.N * a.splits;
  const size_t pbase = (size_t)b * a.N * a.splits;
  const bool staged = npart <= kStagedParts;
  const VocabPartial none{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
  for (int pass = 0; pass < (a.sampling ? 2 : 1); ++pass) {
    const VocabPartial* src = pass == 0 ? a.part : a.part_q;
    if (staged) {
      for (int i = threadIdx.x; i < npart; i += blockDim.x)
        s_stage[i] = __ldcg(reinterpret_cast<const float4*>(src + pbase + i));
      __syncthreads();
    }
    for (int u = threadIdx.x; u < a.N; u += blockDim.x) {
      VocabPartial r = none;
      for (int s2 = 0; s2 < a.splits; ++s2) {
        const int i = u * a.splits + s2;
        const float4 v = staged ? s_stage[i] : __ldcg(reinterpret_cast<const float4*>(src + pbase + i));
        r = partial_merge(r, {v.x, v.y, v.z, __float_as_int(v.w)});
      }
      const size_t r2 = (size_t)b * a.N + u;
      const float l2 = r.m + log2f(r.s);
      if (pass == 0) {
        s_lse2[u] = l2;
        s_am[u] = r.ai;
        if (a.sampling) a.lse2[r2] = l2;  // the sampling walk kernel reads these
        if (a.row_lse) a.row_lse[r2] = l2 * kLn2;
        if (a.row_argmax) a.row_argmax[r2] = r.ai;
      } else {
        s_lse2q[u] = l2;
        a.lse2_q[r2] = l2;
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) a.seq_cnt[b] = 0;
  __syncthreads();
  sequence_epilogue<T>(a, b, s_lse2, s_lse2q, s_am);
}

// ------------------------------------------------------------------------------------
// host side

int verify_splits(int rows, int V) {
  // One wave of 4 resident 256-thread CTAs per SM on 152 SMs, >= 4096 elements per CTA.
  const int target = 152 * 4;
  int s = target / rows;
  int max_by_len = V / 4096;
  if (max_by_len < 1) max_by_len = 1;
  if (s > max_by_len) s = max_by_len;
  if (s > 64) s = 64;
  if (s < 1) s = 1;
  return s;
}

static int verify_chunk(int V, int splits) {
  int c = (V + splits - 1) / splits;
  return (c + 7) / 8 * 8;
}

size_t verify_ws_layout(int B, int N, int V, int sampling, VerifyWs* w) {
  const size_t rows = (size_t)B * N;
  const int splits = verify_splits((int)rows, V);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  VerifyWs l;
  l.splits = splits;
  l.row_cnt = take(rows * 4);
  l.seq_cnt = take((size_t)B * 4);
  l.part = take(rows * splits * sizeof(VocabPartial));
  l.part_q = sampling ? take(rows * splits * sizeof(VocabPartial)) : 0;
  l.lse2 = take(rows * 4);
  l.lse2_q = take(rows * 4);
  l.amax = take(rows * 4);
  l.pc = take(rows * 4);
  l.qc = take(rows * 4);
  l.total = off;
  if (w) *w = l;
  return off;
}

cudaError_t launch_vocab_pass(const void* logits, const void* draft, const int32_t* parent,
                              const int32_t* tokens, int B, int N, int V, tv_dtype dtype, float temperature,
                              char* ws, const VerifyWs& w, int32_t* accepted, int32_t* accept_len,
                              int32_t* bonus, float* p_draft, float* q_draft, float* row_lse,
                              int32_t* row_argmax, int32_t* dev_status, int sampling, cudaStream_t stream) {
  VocabArgs a;
  a.logits = logits;
  a.draft = draft;
  a.parent = parent;
  a.tokens = tokens;
  a.B = B;
  a.N = N;
  a.V = V;
  a.splits = w.splits;
  a.chunk = verify_chunk(V, w.splits);
  a.c2 = kLog2e / temperature;
  a.part = reinterpret_cast<VocabPartial*>(ws + w.part);
  a.part_q = sampling ? reinterpret_cast<VocabPartial*>(ws + w.part_q) : nullptr;
  a.lse2 = reinterpret_cast<float*>(ws + w.lse2);
  a.lse2_q = reinterpret_cast<float*>(ws + w.lse2_q);
  a.amax = reinterpret_cast<int32_t*>(ws + w.amax);
  a.pc = reinterpret_cast<float*>(ws + w.pc);
  a.qc = reinterpret_cast<float*>(ws + w.qc);
  a.row_cnt = reinterpret_cast<unsigned*>(ws + w.row_cnt);
  a.seq_cnt = reinterpret_cast<unsigned*>(ws + w.seq_cnt);
  a.accepted = accepted;
  a.accept_len = accept_len;
  a.bonus = bonus;
  a.p_draft = p_draft;
  a.q_draft = q_draft;
  a.row_lse = row_lse;
  a.row_argmax = row_argmax;
  a.dev_status = dev_status;
  a.sampling = sampling;
  const size_t esz = dtype == TV_BF16 ? 2 : 4;
  bool vec = ((size_t)V * esz) % 16 == 0 && (reinterpret_cast<uintptr_t>(logits) % 16) == 0 &&
             (!sampling || (reinterpret_cast<uintptr_t>(draft) % 16) == 0);
  const unsigned grid = (unsigned)((size_t)B * N * w.splits);
  if (dtype == TV_BF16) {
    if (vec)
      vocab_pass_kernel<uint16_t, true><<<grid, 256, 0, stream>>>(a);
    else
      vocab_pass_kernel<uint16_t, false><<<grid, 256, 0, stream>>>(a);
  } else {
    if (vec)
      vocab_pass_kernel<float, true><<<grid, 256, 0, stream>>>(a);
    else
      vocab_pass_kernel<float, false><<<grid, 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace tv
