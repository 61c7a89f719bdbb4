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
  int32_t* dev_status;
  int sampling;
};

constexpr int kStage = 1024;   // float4 partials staged by a finishing CTA
constexpr int kMaxFinish = 64; // sequences one CTA can finish

__device__ __forceinline__ long long c_first(long long u, const VocabArgs& a) { return u * a.V / a.chunk; }
__device__ __forceinline__ long long c_last(long long u, const VocabArgs& a) {
  return ((u + 1) * a.V - 1) / a.chunk;
}
// number of (row, CTA) partials of sequence b
__device__ __forceinline__ unsigned seq_total(int b, const VocabArgs& a) {
  const long long r0 = (long long)b * a.N, r1 = r0 + a.N - 1;
  const long long distinct = c_last(r1, a) - c_first(r0, a) + 1;
  const long long on_edge = r1 / a.L - r0 / a.L;
  return (unsigned)(distinct + (r1 - r0) - on_edge);
}

struct EpiSmem {
  int* par;
  int* tok;
  float* lse2;
  float* lse2q;
  int* am;
  float4* stage;  // merge staging, reused as match / path afterwards
  float* xc;
  float* yc;
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
  // one round trip: tree, drafted-token logits and (if they fit) every partial
  for (int c = tid; c < N; c += blockDim.x) {
    const int p = a.parent[r0 + c];
    const int t = a.tokens[r0 + c];
    sm.par[c] = p;
    sm.tok[c] = t;
    sm.xc[c] = __ldcg(a.xc + r0 + c);
    if (a.sampling) sm.yc[c] = __ldcg(a.yc + r0 + c);
    const bool ok = (c == 0) ? (p == -1) : (p >= 0 && p < c);
    if (!ok) atomicOr(&s_bad, TV_DEV_BAD_TREE);
    if (c > 0 && (t < 0 || t >= V)) atomicOr(&s_bad, TV_DEV_BAD_TOKEN);
  }
  const VocabPartial none{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
  for (int pass = 0; pass < (a.sampling ? 2 : 1); ++pass) {
    const VocabPartial* src = (pass == 0 ? a.part : a.part_q) + r0 * a.mc;
    if (staged) {
      for (int i = tid; i < nstage; i += blockDim.x) sm.stage[i] = __ldcg(reinterpret_cast<const float4*>(src + i));
      __syncthreads();
    }
    for (int u = tid; u < N; u += blockDim.x) {
      const long long ug = r0 + u;
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
        if (a.row_lse) a.row_lse[ug] = l2 * kLn2;
        if (a.row_argmax) a.row_argmax[ug] = r.ai;
      } else {
        sm.lse2q[u] = l2;
        a.lse2_q[ug] = l2;
      }
    }
    __syncthreads();
  }
  const int bad = s_bad;
  if (bad && tid == 0) set_dev_status(a.dev_status, bad);
  // drafted-token probabilities p_c = 2^(x[parent(c)][t_c] * c2 - lse2[parent(c)])
  for (int c = tid; c < N; c += blockDim.x) {
    float pv = __int_as_float(0x7fc00000), qv = pv;
    if (c > 0 && !bad) {
      const int u = sm.par[c];
      pv = ptx::ex2(fmaf(sm.xc[c], a.c2, -sm.lse2[u]));
      if (a.sampling) qv = ptx::ex2(fmaf(sm.yc[c], a.c2, -sm.lse2q[u]));
    }
    if (a.pc) a.pc[r0 + c] = pv;
    if (a.qc) a.qc[r0 + c] = qv;
    if (a.p_draft) a.p_draft[r0 + c] = pv;
    if (a.q_draft) a.q_draft[r0 + c] = qv;
  }
  if (a.sampling) {
    __syncthreads();
    return;  // the sampling walk runs in its own kernel
  }
  // greedy walk: each node's child whose token equals the node's argmax (lowest index if
  // several) is found in parallel, then the links are followed from the root
  int* match = reinterpret_cast<int*>(sm.stage);
  int* path = match + kMaxNodes;
  for (int c = tid; c < N; c += blockDim.x) match[c] = 0x7fffffff;
  __syncthreads();
  if (!bad)
    for (int c = 1 + tid; c < N; c += blockDim.x)
      if (sm.tok[c] == sm.am[sm.par[c]]) atomicMin(&match[sm.par[c]], c);
  __syncthreads();
  if (tid == 0) {
    int cur = 0, len = 0;
    if (!bad) {
      for (int nxt = match[0]; nxt != 0x7fffffff; nxt = match[cur]) {
        path[len++] = nxt;
        cur = nxt;
      }
    }
    s_len = len;
    s_bonus = bad ? -1 : sm.am[cur];
  }
  __syncthreads();
  const int len = s_len;
  for (int j = tid; j < N; j += blockDim.x) a.accepted[r0 + j] = j < len ? path[j] : -1;
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
  const long long cta = blockIdx.x;
  const long long e0 = cta * a.chunk;
  const long long e1 = min(a.E, e0 + a.chunk);
  const long long u_begin = e0 / a.V, u_end = (e1 - 1) / a.V;
  const T* X = reinterpret_cast<const T*>(a.logits);
  const T* Y = reinterpret_cast<const T*>(a.draft);
  int cur_seq = -1;
  for (long long u = u_begin; u <= u_end; ++u) {
    const int b = (int)(u / a.N);
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
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    // one atomic per sequence this CTA touched; the CTA completing a sequence finishes it
    int nf = 0;
    const int b_first = (int)(u_begin / a.N), b_last = (int)(u_end / a.N);
    for (int b = b_first; b <= b_last; ++b) {
      const long long lo = max(u_begin, (long long)b * a.N), hi = min(u_end, (long long)b * a.N + a.N - 1);
      const unsigned mine = (unsigned)(hi - lo + 1);
      const unsigned prev = atomicAdd(a.seq_cnt + b, mine);
      if (prev + mine == seq_total(b, a) && nf < kMaxFinish) s_finish[nf++] = b;
    }
    s_nfinish = nf;
  }
  __syncthreads();
  const int nf = s_nfinish;
  if (nf == 0) return;
  __threadfence();
  EpiSmem sm{s_par, s_tok, s_lse2, s_lse2q, s_am, s_stage, s_xc, s_yc};
  for (int i = 0; i < nf; ++i) {
    const int b = s_finish[i];
    if (tid == 0) a.seq_cnt[b] = 0;
    sequence_epilogue<T>(a, b, sm);
  }
}

// ------------------------------------------------------------------------------------
// TMA variant (16-byte aligned rows): each CTA bulk-copies its contiguous byte range into
// a ring of shared-memory stages (all stages in flight at once) and reduces from there.

constexpr int kTmaThreads = 512;
constexpr int kPieceBytes = 16384;  // per array per stage
constexpr int kRingBytes = 196608;  // 12 stages (greedy) or 6 double stages (sampling)

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          ptx::smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(ptx::smem_addr(bar))
      : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kTmaThreads, 1) vocab_pass_tma_kernel(VocabArgs a) {
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ VocabPartial red[32];
  __shared__ uint64_t full[12];
  __shared__ int s_par[kMaxNodes];
  __shared__ int s_tok[kMaxNodes];
  __shared__ int s_finish[kMaxFinish];
  __shared__ int s_nfinish;
  __shared__ int s_abort;
  constexpr int kE = kPieceBytes / (int)sizeof(T);  // elements per piece
  const int tid = threadIdx.x;
  const int arrays = a.sampling ? 2 : 1;
  const int nst = kRingBytes / (kPieceBytes * arrays);
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
    ptx::mbar_arrive_expect_tx(&full[st], bytes * arrays);
    unsigned char* dst = ring + (size_t)st * kPieceBytes * arrays;
    bulk_g2s(dst, X + q0, bytes, &full[st]);
    if (arrays == 2) bulk_g2s(dst + kPieceBytes, Y + q0, bytes, &full[st]);
  };
  if (tid == 0) {
    for (int st = 0; st < nst; ++st) ptx::mbar_init(&full[st], 1);
    s_abort = 0;
    ptx::fence_mbar_init();
    for (int pc = 0; pc < min(nst, npieces); ++pc) issue(pc);
  }
  __syncthreads();
  RowAcc acc, accq;
  acc.init();
  accq.init();
  int cur_seq = -1;
  for (int pc = 0; pc < npieces; ++pc) {
    const int st = pc % nst;
    const long long q0 = e0 + (long long)pc * kE;
    const long long q1 = min(e1, q0 + kE);
    bool ok = ptx::mbar_wait(&full[st], (pc / nst) & 1, &s_abort);
    (void)ok;
    const unsigned char* stage = ring + (size_t)st * kPieceBytes * arrays;
    const T* xs = reinterpret_cast<const T*>(stage);
    const T* ys = reinterpret_cast<const T*>(stage + kPieceBytes);
    for (long long u = q0 / a.V; u <= (q1 - 1) / a.V; ++u) {
      const long long rowbase = u * a.V;
      const long long x0 = max(q0, rowbase), x1 = min(q1, rowbase + a.V);
      // 16-byte vectors of the segment [x0, x1) (both ends are multiples of 8 elements)
      const int v_lo = (int)((x0 - q0) * (long long)sizeof(T) / 16);
      const int v_hi = (int)((x1 - q0) * (long long)sizeof(T) / 16);
      constexpr int kN = Vec16<T>::kN;
      for (int j = v_lo + tid; j < v_hi; j += kTmaThreads) {
        const int col = (int)(q0 - rowbase) + j * kN;  // column of the first element
        float xv[kN];
        unpack16<T>(reinterpret_cast<const uint4*>(stage)[j], xv);
        acc.template push<kN>(xv, col, a.c2);
        if (arrays == 2) {
          float yv[kN];
          unpack16<T>(reinterpret_cast<const uint4*>(ys)[j], yv);
          accq.template push<kN>(yv, col, a.c2);
        }
      }
      // drafted tokens of row u that fall in this segment: read them from the stage
      const int b = (int)(u / a.N);
      const int ul = (int)(u - (long long)b * a.N);
      if (b != cur_seq) {
        __syncthreads();
        for (int c = tid; c < a.N; c += kTmaThreads) {
          s_par[c] = a.parent[(size_t)b * a.N + c];
          s_tok[c] = a.tokens[(size_t)b * a.N + c];
        }
        __syncthreads();
        cur_seq = b;
      }
      const int c_lo = (int)(x0 - rowbase), c_hi = (int)(x1 - rowbase);
      for (int c = 1 + tid; c < a.N; c += kTmaThreads) {
        const int t = s_tok[c];
        if (s_par[c] == ul && t >= c_lo && t < c_hi) {
          const int off = (int)(rowbase + t - q0);
          a.xc[(size_t)b * a.N + c] = to_f32(xs[off]);
          if (arrays == 2) a.yc[(size_t)b * a.N + c] = to_f32(ys[off]);
        }
      }
      // this CTA's share of row u ends here: one partial per row and array
      if (x1 == min(e1, rowbase + a.V)) {
        const VocabPartial p = block_merge({acc.mc, acc.s, acc.av, acc.ai}, red);
        VocabPartial pq{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
        if (arrays == 2) pq = block_merge({accq.mc, accq.s, accq.av, accq.ai}, red);
        if (tid == 0) {
          const size_t slot = (size_t)u * a.mc + (size_t)(cta - c_first(u, a));
          a.part[slot] = p;
          if (arrays == 2) a.part_q[slot] = pq;
        }
        acc.init();
        accq.init();
      }
    }
    __syncthreads();  // stage consumed
    if (tid == 0 && pc + nst < npieces) issue(pc + nst);
  }
  if (tid == 0 && s_abort) set_dev_status(a.dev_status, TV_DEV_TIMEOUT);
  __threadfence();
  __syncthreads();
  const long long u_begin = e0 / a.V, u_end = (e1 - 1) / a.V;
  if (tid == 0) {
    int nf = 0;
    const int b_first = (int)(u_begin / a.N), b_last = (int)(u_end / a.N);
    for (int b = b_first; b <= b_last; ++b) {
      const long long lo = max(u_begin, (long long)b * a.N), hi = min(u_end, (long long)b * a.N + a.N - 1);
      const unsigned mine = (unsigned)(hi - lo + 1);
      const unsigned prev = atomicAdd(a.seq_cnt + b, mine);
      if (prev + mine == seq_total(b, a) && nf < kMaxFinish) s_finish[nf++] = b;
    }
    s_nfinish = nf;
  }
  __syncthreads();
  const int nf = s_nfinish;
  if (nf == 0) return;
  __threadfence();
  // the ring is drained: carve the epilogue's arrays from it
  float* e_lse2 = reinterpret_cast<float*>(ring);
  float* e_lse2q = e_lse2 + kMaxNodes;
  int* e_am = reinterpret_cast<int*>(e_lse2q + kMaxNodes);
  float* e_xc = reinterpret_cast<float*>(e_am + kMaxNodes);
  float* e_yc = e_xc + kMaxNodes;
  float4* e_stage = reinterpret_cast<float4*>(e_yc + kMaxNodes);
  EpiSmem sm{s_par, s_tok, e_lse2, e_lse2q, e_am, e_stage, e_xc, e_yc};
  for (int i = 0; i < nf; ++i) {
    const int b = s_finish[i];
    if (tid == 0) a.seq_cnt[b] = 0;
    sequence_epilogue<T>(a, b, sm);
  }
}

// ------------------------------------------------------------------------------------
// host side

constexpr int kVocabThreads = 512;
constexpr long long kMinChunk = 2048;  // elements
constexpr int kGridCap = 4096;         // CTAs (bounds the workspace)
constexpr int kRowsPerCta = 32;        // at most this many rows (+1) per CTA

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
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152 * 4;
  if (!cache[dev]) {
    int per_sm = 0, sms = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vocab_pass_kernel<T, kVec>, kVocabThreads, 0);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = per_sm > 0 && sms > 0 ? per_sm * sms : 152 * 4;
  }
  return cache[dev];
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
}

template <typename T, bool kVec>
static cudaError_t launch_vocab_t(VocabArgs a, cudaStream_t stream) {
  plan_grid(a, resident_ctas<T, kVec>());
  const long long G = (a.E + a.chunk - 1) / a.chunk;
  vocab_pass_kernel<T, kVec><<<(unsigned)G, kVocabThreads, 0, stream>>>(a);
  return cudaSuccess;
}

template <typename T>
static cudaError_t launch_vocab_tma(VocabArgs a, cudaStream_t stream) {
  static bool attr_set[64] = {false};
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(vocab_pass_tma_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kRingBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  plan_grid(a, sms);  // one CTA per SM: the ring takes most of the shared memory
  const long long G = (a.E + a.chunk - 1) / a.chunk;
  vocab_pass_tma_kernel<T><<<(unsigned)G, kTmaThreads, kRingBytes, stream>>>(a);
  return cudaSuccess;
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
