// Fused per-node vocabulary pass and greedy acceptance walk.
//
// Speculative-decoding blog, "greedy decoding, intuitive version" / "acceptance
// probability for sampling": every drafted position needs the target's choice (argmax)
// and the target probability of the drafted token p_u(t).  One streaming, vectorised
// read of the logits yields, per row, the argmax (lowest index among equal raw values)
// and the base-2 log-sum-exp of x/T.
//
// Work split: the B*N*V logits are cut into equal contiguous ranges, one per resident CTA
// (one full wave, identical bytes per CTA).  A CTA writes one partial (max, sum, argmax)
// per row segment it covers and, on the way, the raw logit of every drafted token that
// falls in its range.  The CTA that contributes the last partial of a sequence (one
// atomic per sequence, against a closed-form count) merges that sequence's rows and runs
// its epilogue: drafted-token probabilities and, for greedy verification, the walk.
#include "tv_kernels.cuh"
#include "tv_ptx.cuh"

#include <algorithm>
#include <atomic>

namespace tv {


struct VocabPartial {
  float m;   // max of x * c2 over the chunk (base-2 scaled)
  float s;   // sum 2^(x*c2 - m)
  float av;  // raw max value
  int ai;    // its lowest index
};

// floor(x / d) for x >= 0 whose quotient is below 2^22, without a 64-bit integer
// division: an fp32 estimate x * (1/d) has relative error below 3 * 2^-24, so it is off
// by at most one, which one remainder check corrects.  Every quotient this file takes
// (a row, a sequence, a CTA index) is below 2^18.
struct DivQ {
  long long d;
  float r;
  __device__ __forceinline__ long long operator()(long long x) const {
    long long q = (long long)__float2int_rz(__ll2float_rn(x) * r);
    const long long rem = x - q * d;
    if (rem < 0)
      --q;
    else if (rem >= d)
      ++q;
    return q;
  }
};
inline DivQ make_div(long long d) { return {d, (float)(1.0 / (double)d)}; }

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

// max(a, b, c) in one instruction
__device__ __forceinline__ float vmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
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

// Warp-wide merge of partials in three cheap reductions instead of five pairwise merges:
// the common scaled max first, then every sum rescaled once to it and added, then the
// lowest column among the lanes that hold the raw max.
__device__ __forceinline__ VocabPartial warp_merge(VocabPartial p) {
  float m = p.m, av = p.av;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    av = fmaxf(av, __shfl_xor_sync(0xffffffffu, av, o));
  }
  float s = p.s > 0.f ? p.s * ptx::ex2(p.m - m) : 0.f;
  int ai = p.av == av ? p.ai : 0x7fffffff;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    ai = min(ai, __shfl_xor_sync(0xffffffffu, ai, o));
  }
  return {m, s, av, ai};
}
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

// Accumulate x[v0, v1) of one row into `acc`: 16-byte streaming loads in batches of six
// per thread, the next batch issued before the current one is processed (kVec); scalar
// loads otherwise.
template <typename T, bool kVec>
__device__ __forceinline__ void scan_chunk(const T* __restrict__ row, int v0, int v1, float c2, RowAcc& acc) {
  if constexpr (kVec) {
    constexpr int kN = Vec16<T>::kN;
    constexpr int kBatch = 6;  // 16-byte loads per batch; batches A and B alternate
    const int nvec = (v1 - v0) / kN;
    const uint4* p = reinterpret_cast<const uint4*>(row + v0);
    const int stride = blockDim.x;
    const int step = kBatch * stride;
    uint4 A[kBatch], B[kBatch];
    auto load = [&](uint4* buf, int j) {
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (j + k * stride < nvec) buf[k] = __ldcs(p + j + k * stride);
    };
    auto consume = [&](const uint4* buf, int j) {
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int idx = j + k * stride;
        if (idx < nvec) {
          float x[kN];
          unpack16<T>(buf[k], x);
          acc.template push<kN>(x, v0 + idx * kN, c2);
        }
      }
    };
    int j = threadIdx.x;
    load(A, j);
    for (; j < nvec; j += 2 * step) {
      load(B, j + step);
      consume(A, j);
      load(A, j + 2 * step);
      consume(B, j + step);
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
  int B, N, V;
  long long E;      // B * N * V elements
  long long chunk;  // elements per CTA (multiple of 8)
  long long L;      // chunk / gcd(V, chunk): row boundaries u*V on a chunk edge <=> L | u
  int mc;           // partial slots per row (>= CTAs covering any row)
  DivQ dV, dN, dC, dL;  // division by V, N, chunk and L
  float c2;         // log2(e) / T
  VocabPartial* part;    // [rows][mc]
  VocabPartial* part_q;  // [rows][mc]
  float* lse2;    // [rows] base-2 lse of x*c2 (sampling walk input)
  float* lse2_q;  // [rows]
  float* xc;      // [rows] raw target logit of node c's token in its parent's row
  float* yc;      // [rows] same for the draft logits
  float* pc;      // [rows] p_{parent(c)}(t_c) (fp32), sampling walk input
  float* qc;
  unsigned* seq_cnt;  // [B] completion counters
  // outputs
  int32_t* accepted;
  int32_t* accept_len;
  int32_t* bonus;
  float* p_draft;
  float* q_draft;
  float* row_lse;
  int32_t* row_argmax;
  float* row_lse_q;   // draft rows' natural-log lse (optional)
  int32_t* dev_status;
  int sampling;
};

constexpr int kStage = 1024;   // float4 partials staged by a finishing CTA
constexpr int kMaxFinish = 64; // sequences one CTA can finish
constexpr int kRowsPerCta = 32;                // the host plan gives a CTA at most this many rows (+ 2 partial)
constexpr int kMaxSeg = kRowsPerCta + 4;       // row segments one CTA can cover

__device__ __forceinline__ long long c_first(long long u, const VocabArgs& a) { return a.dC(u * a.V); }
__device__ __forceinline__ long long c_last(long long u, const VocabArgs& a) { return a.dC((u + 1) * a.V - 1); }
// number of (row, CTA) partials of sequence b
__device__ __forceinline__ unsigned seq_total(int b, const VocabArgs& a) {
  const long long r0 = (long long)b * a.N, r1 = r0 + a.N - 1;
  const long long distinct = c_last(r1, a) - c_first(r0, a) + 1;
  const long long on_edge = a.dL(r1) - a.dL(r0);
  return (unsigned)(distinct + (r1 - r0) - on_edge);
}

struct EpiSmem {
  int* par;
  int* tok;
  float* lse2;
  float* lse2q;
  int* am;
  float4* stage;  // merge staging
  float* xc;
  float* yc;
  int* match;  // greedy walk: lowest matching child of each node
  int* path;
};

// Epilogue of sequence b, run by the CTA that wrote its last partial.
template <typename T>
__device__ void sequence_epilogue(const VocabArgs& a, int b, const EpiSmem& sm) {
  __shared__ int s_bad, s_len, s_bonus;
  const int N = a.N, V = a.V, tid = threadIdx.x;
  const long long r0 = (long long)b * N;
  const int nstage = N * a.mc;
  const bool staged = nstage <= kStage;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  // one round trip: tree, drafted-token logits and (if they fit) every target partial,
  // all loads of a thread issued before any of them is used
  const VocabPartial* src0 = a.part + r0 * a.mc;
  for (int base = 0; base < max(N, staged ? nstage : 0); base += blockDim.x) {
    const int c = base + tid;
    const bool tree_item = c < N, stage_item = staged && c < nstage;
    int p = 0, t = 0;
    float x = 0.f, y = 0.f;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tree_item) {
      p = a.parent[r0 + c];
      t = a.tokens[r0 + c];
      x = __ldcg(a.xc + r0 + c);
      if (a.sampling) y = __ldcg(a.yc + r0 + c);
    }
    if (stage_item) v = __ldcg(reinterpret_cast<const float4*>(src0 + c));
    if (tree_item) {
      sm.par[c] = p;
      sm.tok[c] = t;
      sm.xc[c] = x;
      if (a.sampling) sm.yc[c] = y;
      else sm.match[c] = 0x7fffffff;
      // a padding row of a ragged batch (parent -1 after the last node) is no draft:
      // its token is not checked; the rule that padding is trailing is checked below
      const bool ok = (c == 0) ? (p == -1) : (p == -1 || (p >= 0 && p < c));
      if (!ok) atomicOr(&s_bad, TV_DEV_BAD_TREE);
      if (c > 0 && p != -1 && (t < 0 || t >= V)) atomicOr(&s_bad, TV_DEV_BAD_TOKEN);
    }
    if (stage_item) sm.stage[c] = v;
  }
  const VocabPartial none{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
  for (int pass = 0; pass < (a.sampling ? 2 : 1); ++pass) {
    const VocabPartial* src = (pass == 0 ? a.part : a.part_q) + r0 * a.mc;
    if (staged && pass == 1)
      for (int i = tid; i < nstage; i += blockDim.x) sm.stage[i] = __ldcg(reinterpret_cast<const float4*>(src + i));
    __syncthreads();
    for (int u = tid; u < N; u += blockDim.x) {
      const long long ug = r0 + u;
      const bool pad = u > 0 && sm.par[u] == -1;
      if (pass == 0 && u >= 2 && !pad && sm.par[u - 1] == -1) atomicOr(&s_bad, TV_DEV_BAD_TREE);
      const int cover = (int)(c_last(ug, a) - c_first(ug, a) + 1);
      VocabPartial r = none;
      for (int k = 0; k < cover; ++k) {
        const int i = u * a.mc + k;
        const float4 v = staged ? sm.stage[i] : __ldcg(reinterpret_cast<const float4*>(src + i));
        r = partial_merge(r, {v.x, v.y, v.z, __float_as_int(v.w)});
      }
      const float l2 = r.m + log2f(r.s);
      if (pass == 0) {
        sm.lse2[u] = l2;
        sm.am[u] = r.ai;
        if (a.sampling) a.lse2[ug] = l2;  // the sampling walk kernel reads these
        if (a.row_lse) a.row_lse[ug] = pad ? __int_as_float(0x7fc00000) : l2 * kLn2;  // NaN: no row
        if (a.row_argmax) a.row_argmax[ug] = pad ? -1 : r.ai;
      } else {
        sm.lse2q[u] = l2;
        a.lse2_q[ug] = l2;
        if (a.row_lse_q) a.row_lse_q[ug] = pad ? __int_as_float(0x7fc00000) : l2 * kLn2;
      }
    }
    __syncthreads();
  }
  const int bad = s_bad;
  if (bad && tid == 0) set_dev_status(a.dev_status, bad);
  // drafted-token probabilities p_c = 2^(x[parent(c)][t_c] * c2 - lse2[parent(c)]); for
  // greedy verification also each node's child whose token equals the node's argmax
  // (lowest index if several)
  for (int c = tid; c < N; c += blockDim.x) {
    float pv = __int_as_float(0x7fc00000), qv = pv;
    if (c > 0 && !bad && sm.par[c] >= 0) {
      const int u = sm.par[c];
      pv = ptx::ex2(fmaf(sm.xc[c], a.c2, -sm.lse2[u]));
      if (a.sampling)
        qv = ptx::ex2(fmaf(sm.yc[c], a.c2, -sm.lse2q[u]));
      else if (sm.tok[c] == sm.am[u])
        atomicMin(&sm.match[u], c);
    }
    if (a.pc) a.pc[r0 + c] = pv;
    if (a.qc) a.qc[r0 + c] = qv;
    if (a.p_draft) a.p_draft[r0 + c] = pv;
    if (a.q_draft) a.q_draft[r0 + c] = qv;
  }
  __syncthreads();
  // the sampling walk runs in its own kernel; the plain statistics call has no walk
  if (a.sampling || !a.accepted) return;
  // greedy walk: follow the matching links from the root
  if (tid == 0) {
    int cur = 0, len = 0;
    if (!bad) {
      for (int nxt = sm.match[0]; nxt != 0x7fffffff; nxt = sm.match[cur]) {
        sm.path[len++] = nxt;
        cur = nxt;
      }
    }
    s_len = len;
    s_bonus = bad ? -1 : sm.am[cur];
  }
  __syncthreads();
  const int len = s_len;
  for (int j = tid; j < N; j += blockDim.x) a.accepted[r0 + j] = j < len ? sm.path[j] : -1;
  if (tid == 0) {
    a.accept_len[b] = len;
    a.bonus[b] = s_bonus;
  }
  __syncthreads();
}

template <typename T>
__device__ __forceinline__ float load_logit(const void* base, size_t idx) {
  return to_f32(reinterpret_cast<const T*>(base)[idx]);
}

template <typename T, bool kVec>
__global__ void __launch_bounds__(512, 1) vocab_pass_kernel(VocabArgs a) {
  __shared__ VocabPartial red[32];
  __shared__ int s_par[kMaxNodes];
  __shared__ int s_tok[kMaxNodes];
  __shared__ float s_lse2[kMaxNodes];
  __shared__ float s_lse2q[kMaxNodes];
  __shared__ int s_am[kMaxNodes];
  __shared__ float4 s_stage[kStage];
  __shared__ float s_xc[kMaxNodes];
  __shared__ float s_yc[kMaxNodes];
  __shared__ int s_finish[kMaxFinish];
  __shared__ int s_nfinish;
  const int tid = threadIdx.x;
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  const long long cta = blockIdx.x;
  const long long e0 = cta * a.chunk;
  const long long e1 = min(a.E, e0 + a.chunk);
  const long long u_begin = a.dV(e0), u_end = a.dV(e1 - 1);
  const T* X = reinterpret_cast<const T*>(a.logits);
  const T* Y = reinterpret_cast<const T*>(a.draft);
  int cur_seq = -1;
  for (long long u = u_begin; u <= u_end; ++u) {
    const int b = (int)a.dN(u);
    const int ul = (int)(u - (long long)b * a.N);
    if (b != cur_seq) {  // tree of this sequence, to find the children of each row
      __syncthreads();
      for (int c = tid; c < a.N; c += blockDim.x) {
        s_par[c] = a.parent[(size_t)b * a.N + c];
        s_tok[c] = a.tokens[(size_t)b * a.N + c];
      }
      __syncthreads();
      cur_seq = b;
    }
    const long long rowbase = u * a.V;
    const int v0 = (int)(max(e0, rowbase) - rowbase);
    const int v1 = (int)(min(e1, rowbase + a.V) - rowbase);
    RowAcc acc;
    acc.init();
    scan_chunk<T, kVec>(X + rowbase, v0, v1, a.c2, acc);
    const VocabPartial p = block_merge({acc.mc, acc.s, acc.av, acc.ai}, red);
    VocabPartial pq{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
    if (a.sampling) {
      RowAcc accq;
      accq.init();
      scan_chunk<T, kVec>(Y + rowbase, v0, v1, a.c2, accq);
      pq = block_merge({accq.mc, accq.s, accq.av, accq.ai}, red);
    }
    const size_t slot = (size_t)u * a.mc + (size_t)(cta - c_first(u, a));
    if (tid == 0) {
      a.part[slot] = p;
      if (a.sampling) a.part_q[slot] = pq;
    }
    // raw logits of the drafted children of row u whose tokens fall in [v0, v1)
    for (int c = 1 + tid; c < a.N; c += blockDim.x) {
      const int t = s_tok[c];
      if (s_par[c] == ul && t >= v0 && t < v1) {
        a.xc[(size_t)b * a.N + c] = to_f32(X[rowbase + t]);
        if (a.sampling) a.yc[(size_t)b * a.N + c] = to_f32(Y[rowbase + t]);
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    // one atomic per sequence this CTA touched; the CTA completing a sequence finishes it
    int nf = 0;
    const int b_first = (int)a.dN(u_begin), b_last = (int)a.dN(u_end);
    for (int b = b_first; b <= b_last; ++b) {
      const long long lo = max(u_begin, (long long)b * a.N), hi = min(u_end, (long long)b * a.N + a.N - 1);
      const unsigned mine = (unsigned)(hi - lo + 1);
      const unsigned prev = ptx::atom_add_acq_rel_gpu(a.seq_cnt + b, mine);
      if (prev + mine == seq_total(b, a) && nf < kMaxFinish) s_finish[nf++] = b;
    }
    s_nfinish = nf;
  }
  __syncthreads();
  const int nf = s_nfinish;
  if (nf == 0) return;
  // the greedy walk's arrays reuse the sampling-only ones
  EpiSmem sm{s_par, s_tok, s_lse2, s_lse2q, s_am, s_stage, s_xc, s_yc, reinterpret_cast<int*>(s_lse2q),
             reinterpret_cast<int*>(s_yc)};
  for (int i = 0; i < nf; ++i) {
    const int b = s_finish[i];
    if (tid == 0) a.seq_cnt[b] = 0;
    sequence_epilogue<T>(a, b, sm);
  }
}

// ------------------------------------------------------------------------------------
// TMA variant (16-byte aligned rows): each CTA bulk-copies its contiguous byte range into
// a ring of shared-memory stages and reduces from there.  Warps run through the pieces
// independently; the last warp to finish a stage refills it.

constexpr int kTmaThreads = 512;
constexpr int kTmaWarps = kTmaThreads / 32;
constexpr int kRingBytes = 196608;  // 3 stages of 64 KB (one array) or 3 double stages of 32 KB (two)
constexpr int kGroupVec = 4;        // 16-byte vectors per thread reduced in one group
// per array per stage: 64 KB (two groups of four vectors per thread) with one logits
// array, 32 KB (one group) with target and draft arrays; three stages either way
template <int kArrays>
struct Pieces {
  static constexpr int kBytes = kArrays == 1 ? 65536 : 32768;
  static constexpr int kVpt = kBytes / 16 / kTmaThreads;  // vectors per thread per piece
  static constexpr int kStages = kRingBytes / (kBytes * kArrays);
};
constexpr int kMaxStages = 3;

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          ptx::smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(ptx::smem_addr(bar))
      : "memory");
}

// Per-thread running state over one row segment: raw max av, scaled max mc = av*c2 and
// sum of 2^(x*c2 - mc) (two halves, so that packed fp32x2 arithmetic applies).  The
// argmax column is not tracked element by element: the 16-byte vector that holds av and
// its first column are kept, and the column is recovered once, when the segment ends.
template <typename T>
struct StreamAcc {
  static constexpr int kN = Vec16<T>::kN;
  float av;
  float mc;
  float2 s;
  uint4 best;
  int bcol;
  __device__ __forceinline__ void init() {
    av = -INFINITY;
    mc = -INFINITY;
    s = make_float2(0.f, 0.f);
    bcol = -1;
  }
  template <int kM>
  __device__ __forceinline__ void add_sums(const float (&x)[kM], float c2) {
    const float2 cc = make_float2(c2, c2), nm = make_float2(-mc, -mc);
    float2 e[kM / 2];
#pragma unroll
    for (int k = 0; k < kM / 2; ++k) {
      const float2 t = __ffma2_rn(make_float2(x[2 * k], x[2 * k + 1]), cc, nm);
      e[k] = make_float2(ptx::ex2(t.x), ptx::ex2(t.y));
    }
#pragma unroll
    for (int w = 1; w < kM / 2; w *= 2)
#pragma unroll
      for (int k = 0; k + w < kM / 2; k += 2 * w) e[k] = __fadd2_rn(e[k], e[k + w]);
    s = __fadd2_rn(s, e[0]);
  }
  __device__ __forceinline__ void raise(float bv, float c2) {
    const float nmc = bv * c2;
    const float r = ptx::ex2(mc - nmc);
    s.x *= r;
    s.y *= r;
    av = bv;
    mc = nmc;
  }
  // kV vectors; vector v starts at column col0 + v * cstride
  template <int kV>
  __device__ __forceinline__ void pushv(const uint4 (&u)[kV], int col0, int cstride, float c2) {
    float x[kV * kN];
    float bm[kV];
#pragma unroll
    for (int v = 0; v < kV; ++v) {
      unpack16<T>(u[v], x + v * kN);
      // vector maximum with three-input max instructions
      float m = x[v * kN];
      int k = 1;
#pragma unroll
      for (; k + 1 < kN; k += 2) m = vmax3(m, x[v * kN + k], x[v * kN + k + 1]);
      if (k < kN) m = fmaxf(m, x[v * kN + k]);
      bm[v] = m;
    }
    float bv = bm[0];
    {
      int v = 1;
#pragma unroll
      for (; v + 1 < kV; v += 2) bv = vmax3(bv, bm[v], bm[v + 1]);
      if (v < kV) bv = fmaxf(bv, bm[v]);
    }
    if (bv == -INFINITY) return;  // all -inf: nothing to add
    if (bv > av) {                // rare: keep the first vector that holds the new max
      bool found = false;
#pragma unroll
      for (int v = 0; v < kV; ++v)
        if (!found && bm[v] == bv) {
          found = true;
          best = u[v];
          bcol = col0 + v * cstride;
        }
      raise(bv, c2);
    }
    add_sums<kV * kN>(x, c2);
  }
  __device__ __forceinline__ void push1(const uint4& u, int col, float c2) {
    float x[kN];
    unpack16<T>(u, x);
    float bv = x[0];
#pragma unroll
    for (int k = 1; k < kN; ++k) bv = fmaxf(bv, x[k]);
    if (bv == -INFINITY) return;
    if (bv > av) {
      best = u;
      bcol = col;
      raise(bv, c2);
    }
    add_sums<kN>(x, c2);
  }
  __device__ __forceinline__ VocabPartial partial() const {
    int ai = 0x7fffffff;
    if (bcol >= 0) {
      float x[kN];
      unpack16<T>(best, x);
#pragma unroll
      for (int k = kN - 1; k >= 0; --k)
        if (x[k] == av) ai = bcol + k;
    }
    return {mc, s.x + s.y, av, ai};
  }
};

template <typename T, int kArrays>
__global__ void __launch_bounds__(kTmaThreads, 1) vocab_pass_tma_kernel(VocabArgs a) {
  extern __shared__ __align__(128) unsigned char ring[];
  constexpr int kPieceBytes = Pieces<kArrays>::kBytes;
  constexpr int kVpt = Pieces<kArrays>::kVpt;
  static_assert(Pieces<kArrays>::kStages == kMaxStages, "three stages");
  __shared__ uint64_t full[kMaxStages];
  __shared__ int s_done[kMaxStages];
  __shared__ VocabPartial s_wp[kArrays][kMaxSeg][kTmaWarps];  // per-warp partials of each row segment
  __shared__ long long s_segslot[kMaxSeg];
  __shared__ int s_finish[kMaxFinish];
  __shared__ unsigned s_total[kMaxFinish];
  __shared__ int s_nfinish;
  __shared__ int s_abort;
  constexpr int kE = kPieceBytes / (int)sizeof(T);  // elements per piece (a power of two)
  constexpr int kN = Vec16<T>::kN;                  // elements per 16-byte vector
  constexpr int nst = kMaxStages;
  static_assert(kVpt * 16 * kTmaThreads == kPieceBytes, "a piece is kVpt vectors per thread");
  static_assert(kMaxNodes <= 2 * kTmaThreads + 1, "each thread owns at most two children");
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  const long long cta = blockIdx.x;
  const long long e0 = cta * a.chunk;
  const long long e1 = min(a.E, e0 + a.chunk);
  const int npieces = (int)((e1 - e0 + kE - 1) / kE);
  const T* X = reinterpret_cast<const T*>(a.logits);
  const T* Y = reinterpret_cast<const T*>(a.draft);
  auto issue = [&](int piece) {
    const int st = piece % nst;
    const long long q0 = e0 + (long long)piece * kE;
    const uint32_t bytes = (uint32_t)((min(e1, q0 + kE) - q0) * (long long)sizeof(T));
    ptx::mbar_arrive_expect_tx(&full[st], bytes * kArrays);
    unsigned char* dst = ring + (size_t)st * kPieceBytes * kArrays;
    bulk_g2s(dst, X + q0, bytes, &full[st]);
    if (kArrays == 2) bulk_g2s(dst + kPieceBytes, Y + q0, bytes, &full[st]);
  };
  const long long u_begin = a.dV(e0), u_end = a.dV(e1 - 1);
  const int b_first = (int)a.dN(u_begin), b_last = (int)a.dN(u_end);
  // Drafted-token logits: the thread owning child c (c = 1 + tid + k * kTmaThreads) reads
  // x[parent row][token] from the stage of the piece that holds it, if this CTA's range does.
  int cap_pc[2], cap_off[2], tp[2], tt[2];
  auto fetch_tree = [&](int bs) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int c = 1 + tid + k * kTmaThreads;
      tp[k] = c < a.N ? a.parent[(size_t)bs * a.N + c] : -1;
      tt[k] = c < a.N ? a.tokens[(size_t)bs * a.N + c] : -1;
    }
  };
  auto make_caps = [&](int bs) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      cap_pc[k] = -1;
      cap_off[k] = 0;
      // malformed trees are reported by the epilogue
      if (tp[k] >= 0 && tp[k] < a.N && tt[k] >= 0 && tt[k] < a.V) {
        const long long g = ((long long)bs * a.N + tp[k]) * a.V + tt[k];
        if (g >= e0 && g < e1) {
          cap_pc[k] = (int)((g - e0) / kE);
          cap_off[k] = (int)((g - e0) % kE);
        }
      }
    }
  };
  // a capture is retired once taken, so that the next piece to stop at is the earliest
  // of the captures still pending (a thread owns two children when N > 513)
  auto capture = [&](int pc, int bs, const unsigned char* stage) {
#pragma unroll
    for (int k = 0; k < 2; ++k)
      if (cap_pc[k] == pc) {
        const size_t c = (size_t)bs * a.N + 1 + tid + k * kTmaThreads;
        a.xc[c] = to_f32(reinterpret_cast<const T*>(stage)[cap_off[k]]);
        if (kArrays == 2) a.yc[c] = to_f32(reinterpret_cast<const T*>(stage + kPieceBytes)[cap_off[k]]);
        cap_pc[k] = -1;
      }
  };
  fetch_tree(b_first);  // issued ahead of the bulk copies, so that it does not queue behind them
  if (tid == 0) {
    for (int st = 0; st < nst; ++st) {
      ptx::mbar_init(&full[st], 1);
      s_done[st] = 0;
    }
    s_abort = 0;
    ptx::fence_mbar_init();
    for (int pc = 0; pc < min(nst, npieces); ++pc) issue(pc);
  } else if (tid >= 32 && tid < 64) {
    for (int i = lane; i < min(b_last - b_first + 1, kMaxFinish); i += 32) s_total[i] = seq_total(b_first + i, a);
  }
  __syncthreads();
  make_caps(b_first);
  StreamAcc<T> acc, accq;
  acc.init();
  accq.init();
  // current row u: [rowbase, row_end) in flat element indices; rowbase <= q0 < row_end
  // holds at the start of every piece
  long long u = u_begin, rowbase = u_begin * a.V, row_end = rowbase + a.V;
  int b = b_first, ul = (int)(u_begin - (long long)b_first * a.N);
  long long slot = u_begin * a.mc + (cta - c_first(u_begin, a));
  // Where this CTA's share of row u ends, every warp parks its merged partial in shared
  // memory (no block barrier in the streaming loop); the segments are merged at the end.
  int seg = 0;
  auto row_done = [&]() {
    const VocabPartial p = warp_merge(acc.partial());
    VocabPartial pq{};
    if (kArrays == 2) pq = warp_merge(accq.partial());
    if (seg < kMaxSeg) {
      if (lane == 0) {
        s_wp[0][seg][wid] = p;
        if (kArrays == 2) s_wp[kArrays - 1][seg][wid] = pq;
      }
      if (tid == 0) s_segslot[seg] = slot;
    }
    ++seg;
    acc.init();
    accq.init();
  };
  auto next_row = [&]() {  // row u + 1 starts inside this CTA's range: its first partial slot
    rowbase = row_end;
    row_end += a.V;
    ++u;
    slot = u * a.mc;
    if (++ul == a.N) {
      ul = 0;
      ++b;
      fetch_tree(b);
      make_caps(b);
    }
  };
  int st = 0;
  uint32_t phase = 0;
  long long q0 = e0;
  // fast-path bookkeeping in 32 bits: elements from the piece start to the end of row u
  int rem = (int)(row_end - q0);
  const bool last_full = (e1 - e0) % kE == 0;
  int next_cap = min((unsigned)cap_pc[0], (unsigned)cap_pc[1]);  // -1 (none) sorts last
  for (int pc = 0; pc < npieces; ++pc, q0 += kE) {
    ptx::mbar_wait(&full[st], phase, &s_abort);
    const unsigned char* stage = ring + (size_t)st * kPieceBytes * kArrays;
    const uint4* xv4 = reinterpret_cast<const uint4*>(stage);
    const uint4* yv4 = reinterpret_cast<const uint4*>(stage + kPieceBytes);
    if (rem >= kE && (pc + 1 < npieces || last_full)) {
      // the whole piece lies in row u: vectors tid + v * kTmaThreads of every array
      const int col0 = (a.V - rem) + tid * kN;
      // groups of four vectors per thread: vectors tid + v * kTmaThreads
#pragma unroll
      for (int g0 = 0; g0 < kVpt; g0 += kGroupVec) {
        uint4 u[kGroupVec];
#pragma unroll
        for (int v = 0; v < kGroupVec; ++v) u[v] = xv4[tid + (g0 + v) * kTmaThreads];
        acc.template pushv<kGroupVec>(u, col0 + g0 * kTmaThreads * kN, kTmaThreads * kN, a.c2);
        if (kArrays == 2) {
#pragma unroll
          for (int v = 0; v < kGroupVec; ++v) u[v] = yv4[tid + (g0 + v) * kTmaThreads];
          accq.template pushv<kGroupVec>(u, col0 + g0 * kTmaThreads * kN, kTmaThreads * kN, a.c2);
        }
      }
      if (pc == next_cap) capture(pc, b, stage);
      rem -= kE;
      if (rem == 0) {
        row_done();
        if (q0 + kE < e1) {
          next_row();
          rem = a.V;
        }
      }
    } else {
      const long long q1 = min(e1, q0 + kE);
      for (;;) {
        const long long x0 = max(q0, rowbase), x1 = min(q1, row_end);
        const int col0 = (int)(q0 - rowbase);
        // 16-byte vectors of the segment [x0, x1) (both ends are multiples of 8 elements)
        const int v_lo = (int)((x0 - q0) / kN), v_hi = (int)((x1 - q0) / kN);
        for (int j = v_lo + tid; j < v_hi; j += kTmaThreads) {
          acc.push1(xv4[j], col0 + j * kN, a.c2);
          if (kArrays == 2) accq.push1(yv4[j], col0 + j * kN, a.c2);
        }
        capture(pc, b, stage);
        if (x1 == min(e1, row_end)) row_done();
        if (row_end > q1 || row_end >= e1) break;  // row u continues in the next piece
        next_row();
      }
      rem = (int)(row_end - (q0 + kE));
    }
    next_cap = min((unsigned)cap_pc[0], (unsigned)cap_pc[1]);
    // stage consumed by this warp; the last warp through refills it
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&s_done[st], 1) == kTmaWarps - 1) {
        __threadfence_block();
        s_done[st] = 0;
        if (pc + nst < npieces) {
          ptx::fence_proxy_async_smem();
          issue(pc + nst);
        }
      }
    }
    if (++st == nst) {
      st = 0;
      phase ^= 1;
    }
  }
  __syncthreads();
  // one partial per (row segment, array): merge the warps' partials
  for (int sg = wid; sg < min(seg, kMaxSeg); sg += kTmaWarps) {
#pragma unroll
    for (int ar = 0; ar < kArrays; ++ar) {
      VocabPartial q = lane < kTmaWarps ? s_wp[ar][sg][lane] : VocabPartial{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
      q = warp_merge(q);
      if (lane == 0) (ar == 0 ? a.part : a.part_q)[s_segslot[sg]] = q;
    }
  }
  __syncthreads();
  if (tid == 0) {
    if (s_abort) set_dev_status(a.dev_status, TV_DEV_TIMEOUT);
    if (seg > kMaxSeg) set_dev_status(a.dev_status, TV_DEV_BAD_TREE);  // excluded by the host plan
    int nf = 0;
    for (int bb = b_first; bb <= b_last; ++bb) {
      const long long lo = max(u_begin, (long long)bb * a.N), hi = min(u_end, (long long)bb * a.N + a.N - 1);
      const unsigned mine = (unsigned)(hi - lo + 1);
      const unsigned prev = ptx::atom_add_acq_rel_gpu(a.seq_cnt + bb, mine);
      const int i = bb - b_first;
      if (i < kMaxFinish && prev + mine == s_total[i] && nf < kMaxFinish) s_finish[nf++] = bb;
    }
    s_nfinish = nf;
  }
  __syncthreads();
  const int nf = s_nfinish;
  if (nf == 0) return;
  // the ring is drained: carve the epilogue's arrays from it
  int* e_par = reinterpret_cast<int*>(ring);
  int* e_tok = e_par + kMaxNodes;
  float* e_lse2 = reinterpret_cast<float*>(e_tok + kMaxNodes);
  float* e_lse2q = e_lse2 + kMaxNodes;
  int* e_am = reinterpret_cast<int*>(e_lse2q + kMaxNodes);
  float* e_xc = reinterpret_cast<float*>(e_am + kMaxNodes);
  float* e_yc = e_xc + kMaxNodes;
  int* e_match = reinterpret_cast<int*>(e_yc + kMaxNodes);
  int* e_path = e_match + kMaxNodes;
  float4* e_stage = reinterpret_cast<float4*>(e_path + kMaxNodes);
  EpiSmem sm{e_par, e_tok, e_lse2, e_lse2q, e_am, e_stage, e_xc, e_yc, e_match, e_path};
  for (int i = 0; i < nf; ++i) {
    const int bs = s_finish[i];
    if (tid == 0) a.seq_cnt[bs] = 0;
    sequence_epilogue<T>(a, bs, sm);
  }
}

// ------------------------------------------------------------------------------------
// host side

constexpr int kVocabThreads = 512;
constexpr long long kMinChunk = 2048;  // elements
constexpr int kGridCap = 4096;         // CTAs (bounds the workspace)

static long long gcd_ll(long long x, long long y) {
  while (y) {
    const long long t = x % y;
    x = y;
    y = t;
  }
  return x;
}

// partial slots per row for any grid of at most kGridCap CTAs
static int ws_mc(long long rows) { return (int)((kGridCap + rows - 1) / rows) + 2; }

int verify_slots_per_row(int rows) { return ws_mc(rows); }

size_t verify_ws_layout(int B, int N, int V, int sampling, VerifyWs* w) {
  const size_t rows = (size_t)B * N;
  const int mc = ws_mc((long long)rows);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  VerifyWs l;
  l.splits = mc;
  l.row_cnt = 0;  // counter region: [row_cnt, part)
  l.seq_cnt = take((size_t)B * 4);
  l.part = take(rows * mc * sizeof(VocabPartial));
  l.part_q = sampling ? take(rows * mc * sizeof(VocabPartial)) : 0;
  l.lse2 = take(rows * 4);
  l.lse2_q = take(rows * 4);
  l.xc = take(rows * 4);  // raw drafted-token logits (target)
  l.pc = take(rows * 4);
  l.qc = take(rows * 4);
  l.yc = take(rows * 4);    // raw drafted-token logits (draft)
  l.total = off;
  if (w) *w = l;
  (void)V;
  return off;
}

template <typename T, bool kVec>
static int resident_ctas() {
  static std::atomic<int> cache[64];  // 0 = not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152 * 4;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (!n) {
    int per_sm = 0, sms = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vocab_pass_kernel<T, kVec>, kVocabThreads, 0);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    n = per_sm > 0 && sms > 0 ? per_sm * sms : 152 * 4;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

static void plan_grid(VocabArgs& a, long long G) {
  const long long rows = (long long)a.B * a.N;
  G = std::min<long long>({G, (long long)kGridCap, (a.E + kMinChunk - 1) / kMinChunk});
  G = std::max<long long>(G, (rows + kRowsPerCta - 1) / kRowsPerCta);  // bounds sequences finished per CTA
  if (G < 1) G = 1;
  long long chunk = (a.E + G - 1) / G;
  chunk = (chunk + 7) / 8 * 8;
  a.chunk = chunk;
  a.L = chunk / gcd_ll((long long)a.V, chunk);
  a.mc = (int)((a.V + chunk - 1) / chunk) + 1;
  a.dV = make_div(a.V);
  a.dN = make_div(a.N);
  a.dC = make_div(a.chunk);
  a.dL = make_div(a.L);
}

template <typename T, bool kVec>
static cudaError_t launch_vocab_t(VocabArgs a, cudaStream_t stream) {
  plan_grid(a, resident_ctas<T, kVec>());
  const long long G = (a.E + a.chunk - 1) / a.chunk;
  return launch_pdl(vocab_pass_kernel<T, kVec>, dim3((unsigned)G), dim3(kVocabThreads), 0, stream, nullptr, 0, a);
}

template <typename T, int kArrays>
static cudaError_t launch_vocab_tma(VocabArgs a, cudaStream_t stream) {
  static std::atomic<bool> attr_set[64];  // false until the attribute is set on that device
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(vocab_pass_tma_kernel<T, kArrays>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sm_share_verify() > 0) sms = std::min(sms, sm_share_verify());
  plan_grid(a, sms);  // one CTA per SM: the ring takes most of the shared memory
  const long long G = (a.E + a.chunk - 1) / a.chunk;
  return launch_pdl(vocab_pass_tma_kernel<T, kArrays>, dim3((unsigned)G), dim3(kTmaThreads), kRingBytes, stream,
                    nullptr, 0, a);
}

template <typename T>
static cudaError_t launch_vocab_tma(VocabArgs a, cudaStream_t stream) {
  return a.sampling ? launch_vocab_tma<T, 2>(a, stream) : launch_vocab_tma<T, 1>(a, stream);
}

cudaError_t launch_vocab_pass(const void* logits, const void* draft, const int32_t* parent,
                              const int32_t* tokens, int B, int N, int V, tv_dtype dtype, float temperature,
                              char* ws, const VerifyWs& w, int32_t* accepted, int32_t* accept_len,
                              int32_t* bonus, float* p_draft, float* q_draft, float* row_lse,
                              int32_t* row_argmax, float* row_lse_q, int32_t* dev_status, int sampling,
                              cudaStream_t stream) {
  VocabArgs a;
  a.logits = logits;
  a.draft = draft;
  a.parent = parent;
  a.tokens = tokens;
  a.B = B;
  a.N = N;
  a.V = V;
  a.E = (long long)B * N * V;
  a.c2 = kLog2e / temperature;
  a.part = reinterpret_cast<VocabPartial*>(ws + w.part);
  a.part_q = sampling ? reinterpret_cast<VocabPartial*>(ws + w.part_q) : nullptr;
  a.lse2 = reinterpret_cast<float*>(ws + w.lse2);
  a.lse2_q = reinterpret_cast<float*>(ws + w.lse2_q);
  a.xc = reinterpret_cast<float*>(ws + w.xc);
  a.yc = reinterpret_cast<float*>(ws + w.yc);
  a.pc = reinterpret_cast<float*>(ws + w.pc);
  a.qc = reinterpret_cast<float*>(ws + w.qc);
  a.seq_cnt = reinterpret_cast<unsigned*>(ws + w.seq_cnt);
  a.accepted = accepted;
  a.accept_len = accept_len;
  a.bonus = bonus;
  a.p_draft = p_draft;
  a.q_draft = q_draft;
  a.row_lse = row_lse;
  a.row_argmax = row_argmax;
  a.row_lse_q = row_lse_q;
  a.dev_status = dev_status;
  a.sampling = sampling;
  const size_t esz = dtype == TV_BF16 ? 2 : 4;
  const bool vec = ((size_t)V * esz) % 16 == 0 && (reinterpret_cast<uintptr_t>(logits) % 16) == 0 &&
                   (!sampling || (reinterpret_cast<uintptr_t>(draft) % 16) == 0);
  cudaError_t e;
  if (dtype == TV_BF16)
    e = vec ? launch_vocab_tma<uint16_t>(a, stream) : launch_vocab_t<uint16_t, false>(a, stream);
  else
    e = vec ? launch_vocab_tma<float>(a, stream) : launch_vocab_t<float, false>(a, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace tv
