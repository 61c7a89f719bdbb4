// Tree-masked GQA attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// PTD §3.1: node i attends to the committed prefix and to its observable set pi(i);
// TAPS §4.1: the selected subtree is verified by the target in one pass with tree
// attention.  One CTA owns a tile of 128 query rows that share one KV head: the G query
// heads of a GQA group times NT = 128/G consecutive tree nodes (head-major rows), so each
// K/V tile fetched from HBM by TMA is used by every node and every head of the group.
// The key range [0, P + last node of the tile) is cut into KV splits across CTAs.
//
// Per CTA, warp-specialised:
//   warp 0      TMA producers: lane 0 loads the Q tile once, then K tiles of 128 keys
//               into a 3-slot ring; lane 1 loads the V tiles into a 2-slot ring
//   warp 1      TMEM owner; lane 0 issues S[t&1] = Q K_t^T (M=128, N=128, K=D, fp32
//               in TMEM) as soon as a K tile and an S buffer are free
//   warp 10     lane 0 issues O += P_t V_t (M=128, N=D, K=128, fp32 in TMEM, P_t read
//               from TMEM) as soon as the softmax has written P_t
//   warps 2..9  softmax: two threads per row (each half of a tile's 128 keys); read S
//               from TMEM, apply the tree mask, agree on the row max with the partner
//               thread, keep a running reference max (rescale O only when the max grows
//               by more than 2^8), write P (bf16) into one of two TMEM buffers, so the
//               exponentials of tile t overlap the PV product of tile t-1.
// TMEM columns: S[0] 0..127, S[1] 128..255, O 256..256+D, P[0] 384..447, P[1] 448..511.
// With one split the epilogue normalises O and stores bf16.  With several, the splits of
// a row tile run as one thread-block cluster: each CTA parks its unnormalised O and
// (m, l) in its own shared memory and, after a cluster barrier, merges a slice of the
// rows by reading its peers' partials over distributed shared memory.
#include <cuda.h>

#include <algorithm>

#include "tv_kernels.cuh"
#include "tv_ptx.cuh"

namespace tv {

constexpr int kRows = 128;     // MMA M: query rows per CTA
constexpr int kBN = 128;       // keys per KV tile (MMA N of QK^T, K of PV)
constexpr int kKSlots = 3;     // K ring depth (tiles of 128 keys)
constexpr int kVSlots = 2;     // V ring depth
constexpr int kThreads = 352;  // 11 warps: TMA producers, S issuer, 8 softmax warps, PV issuer
constexpr float kRescaleLog2 = 8.f;
constexpr int kMaxSplits = 8;  // KV splits of a row tile = one portable-size cluster

template <int D>
struct TcCfg {
  static constexpr int kDB = D / 64;                  // 64-element (128-byte) column blocks
  static constexpr int kQBlock = kRows * 128;         // bytes per column block of Q
  static constexpr int kKVBlock = kBN * 128;          // bytes per column block of a K or V tile
  static constexpr int kQBytes = kDB * kQBlock;
  static constexpr int kTileBytes = kDB * kKVBlock;   // one K or V tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kKSlots * kTileBytes;
  static constexpr int kOffPar = kOffV + kVSlots * kTileBytes;
  static constexpr int kOffBar = kOffPar + kMaxNodes * 4;
  static constexpr int kSmemUsed = kOffBar + 256;
  static constexpr int kSmemAlloc = kSmemUsed + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 2 * kBN;           // after S[0], S[1]
  static constexpr uint32_t kColP = 384;               // P[0], P[1]: 64 columns each
  static_assert(kColO + D <= kColP && kColP + 2 * (kBN / 2) <= kTmemCols, "TMEM budget");
  static_assert(kOffV - kOffK >= D * kRows * 4 + kRows * 8, "split partials fit in the drained K ring");
};

struct TcArgs {
  void* out;
  const int32_t* parent;
  int B, Hq, Hkv, N, P, G, NT, MT, splits;
  float c;  // softmax scale * log2(e)
  int32_t* dev_status;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kKSlots];
  uint64_t k_empty[kKSlots];
  uint64_t v_full[kVSlots];
  uint64_t v_empty[kVSlots];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];  // PV(t) complete, on barrier t & 1
  uint64_t o_done;
  uint64_t s_done;
  uint32_t tmem_base;
  int abort;
};

// 64-bit visibility mask of keys [j0, j0 + 64) for tree node `node` (half a KV tile).
__device__ __forceinline__ uint64_t key_mask(int j0, int P, int N, int node, const int* s_par) {
  if (j0 + 64 <= P) return ~0ull;
  uint64_t vis = 0;
  if (j0 < P) vis = (1ull << (P - j0)) - 1ull;
  int a = node, guard = 0;
  while (a >= 0 && guard <= N) {
    const int j = P + a - j0;
    if (j >= 0 && j < 64) vis |= 1ull << j;
    const int pa = s_par[a];
    if (pa >= a) break;  // malformed (flagged when loaded)
    a = pa;
    ++guard;
  }
  return vis;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, TcArgs a) {
  using C = TcCfg<D>;
  extern __shared__ unsigned char smem_raw[];
  __shared__ float s_xmax[2][2][kRows];  // [tile parity][half][row] partial row maxima
  __shared__ float s_xl[2][kRows];       // [half][row] partial row sums
  const uint32_t mis = ptx::smem_addr(smem_raw) & 1023u;
  unsigned char* sm = smem_raw + ((1024u - mis) & 1023u);
  unsigned char* sQ = sm + C::kOffQ;
  unsigned char* sK = sm + C::kOffK;
  unsigned char* sV = sm + C::kOffV;
  int* s_par = reinterpret_cast<int*>(sm + C::kOffPar);
  Bars* bars = reinterpret_cast<Bars*>(sm + C::kOffBar);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the splits of one row tile are consecutive in x and form one cluster (rank = split)
  const int mt = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
  const int hk = blockIdx.y, b = blockIdx.z;
  const int i0 = mt * a.NT;
  const int nodes_hi = min(a.N, i0 + a.NT);
  const int ltot = a.P + nodes_hi;
  const int t_all = (ltot + kBN - 1) / kBN;
  const int tps = (t_all + a.splits - 1) / a.splits;
  const int t_begin = split * tps;
  const int nt = max(0, min(t_all, t_begin + tps) - t_begin);
  const int rows_used = a.G * a.NT;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kKSlots; ++s) {
      ptx::mbar_init(&bars->k_full[s], 1);
      ptx::mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < kVSlots; ++s) {
      ptx::mbar_init(&bars->v_full[s], 1);
      ptx::mbar_init(&bars->v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bars->s_full[s], 1);
      ptx::mbar_init(&bars->s_free[s], 8);
      ptx::mbar_init(&bars->p_full[s], 8);
      ptx::mbar_init(&bars->pv_done[s], 1);
    }
    ptx::mbar_init(&bars->o_done, 1);
    ptx::mbar_init(&bars->s_done, 1);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bars->tmem_base, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp >= 2) {
    // parent array for the mask; zero the Q rows that no TMA box fills
    const int t = threadIdx.x - 64;
    int bad = 0;
    for (int c = t; c < a.N; c += kThreads - 64) {
      const int p = a.parent[(size_t)b * a.N + c];
      s_par[c] = p;
      if (!((c == 0) ? (p == -1) : (p >= 0 && p < c))) bad = 1;
    }
    if (bad) set_dev_status(a.dev_status, TV_DEV_BAD_TREE);
    for (int r = rows_used + t; r < kRows; r += kThreads - 64)
      for (int db = 0; db < C::kDB; ++db) {
        uint4* row = reinterpret_cast<uint4*>(sQ + db * C::kQBlock + r * 128);
#pragma unroll
        for (int k = 0; k < 8; ++k) row[k] = make_uint4(0, 0, 0, 0);
      }
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ producers
    if (lane == 0 && nt > 0) {
      // Q once, then the K tiles; a slot is refilled once S of its previous tile is done
      int issued[kKSlots];
#pragma unroll
      for (int s = 0; s < kKSlots; ++s) issued[s] = 0;
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(rows_used * 128 * C::kDB));
      for (int g = 0; g < a.G; ++g)
        for (int db = 0; db < C::kDB; ++db)
          ptx::tma_load_3d(sQ + db * C::kQBlock + g * a.NT * 128, &tmQ, &bars->q_full, db * 64, i0,
                           b * a.Hq + hk * a.G + g);
      for (int t = 0; t < nt; ++t) {
        const int ks = t % kKSlots;
        if (t >= kKSlots && !ptx::mbar_wait(&bars->k_empty[ks], ((t / kKSlots) - 1) & 1, abort_flag)) break;
        unsigned char* dst = sK + ks * C::kTileBytes;
        const int j0 = (t_begin + t) * kBN;
        ptx::mbar_arrive_expect_tx(&bars->k_full[ks], (uint32_t)C::kTileBytes);
        for (int db = 0; db < C::kDB; ++db)
          ptx::tma_load_3d(dst + db * C::kKVBlock, &tmK, &bars->k_full[ks], db * 64, j0, b * a.Hkv + hk);
        ++issued[ks];
      }
      // never leave the CTA with copies in flight
      ptx::mbar_wait(&bars->q_full, 0, abort_flag);
      for (int s = 0; s < kKSlots; ++s)
        if (issued[s]) ptx::mbar_wait(&bars->k_full[s], (issued[s] - 1) & 1, abort_flag);
    } else if (lane == 1 && nt > 0) {
      // the V tiles; a slot is refilled once PV of its previous tile is done
      int issued[kVSlots];
#pragma unroll
      for (int s = 0; s < kVSlots; ++s) issued[s] = 0;
      ptx::prefetch_tmap(&tmV);
      for (int t = 0; t < nt; ++t) {
        const int vs = t % kVSlots;
        if (t >= kVSlots && !ptx::mbar_wait(&bars->v_empty[vs], ((t / kVSlots) - 1) & 1, abort_flag)) break;
        unsigned char* dst = sV + vs * C::kTileBytes;
        const int j0 = (t_begin + t) * kBN;
        ptx::mbar_arrive_expect_tx(&bars->v_full[vs], (uint32_t)C::kTileBytes);
        for (int db = 0; db < C::kDB; ++db)
          ptx::tma_load_3d(dst + db * C::kKVBlock, &tmV, &bars->v_full[vs], db * 64, j0, b * a.Hkv + hk);
        ++issued[vs];
      }
      for (int s = 0; s < kVSlots; ++s)
        if (issued[s]) ptx::mbar_wait(&bars->v_full[s], (issued[s] - 1) & 1, abort_flag);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      if (nt > 0 && ptx::mbar_wait(&bars->q_full, 0, abort_flag)) {
        constexpr uint32_t idS = ptx::idesc_bf16(kRows, kBN, false, false);
        const uint32_t qaddr = ptx::smem_addr(sQ);
        bool ok = true;
        auto issue_s = [&](int t) -> bool {
          const int ks = t % kKSlots, sb = t & 1;
          if (!ptx::mbar_wait(&bars->k_full[ks], (t / kKSlots) & 1, abort_flag)) return false;
          if (t >= 2 && !ptx::mbar_wait(&bars->s_free[sb], ((t >> 1) - 1) & 1, abort_flag)) return false;
          ptx::tc_fence_after();
          const uint32_t kaddr = ptx::smem_addr(sK + ks * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk & 3) * 32;  // 16-element K step inside a 128-byte row
            const uint64_t ad = ptx::sdesc_sw128(qaddr + (kk >> 2) * C::kQBlock + off, 16, 1024);
            const uint64_t bd = ptx::sdesc_sw128(kaddr + (kk >> 2) * C::kKVBlock + off, 16, 1024);
            ptx::mma_bf16_ss(tmem + sb * kBN, ad, bd, idS, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit(&bars->s_full[sb]);
          ptx::mma_commit(&bars->k_empty[ks]);
          return true;
        };
        // S = QK^T tiles run ahead of the softmax (bounded by the two S buffers); the PV
        // products are issued by warp 10, so neither waits behind the other's issue
        for (int t = 0; ok && t < nt; ++t) ok = issue_s(t);
      }
      ptx::mma_commit(&bars->s_done);
      ptx::mbar_wait(&bars->s_done, 0, abort_flag);
    }
    __syncwarp();
  } else if (warp == kThreads / 32 - 1) {
    // ------------------------------------------------------------------ PV issuer
    if (lane == 0) {
      if (nt > 0) {
        constexpr uint32_t idO = ptx::idesc_bf16(kRows, D, false, true);
        for (int t = 0; t < nt; ++t) {
          const int vs = t % kVSlots, pb = t & 1;
          if (!ptx::mbar_wait(&bars->p_full[pb], (t >> 1) & 1, abort_flag)) break;
          if (!ptx::mbar_wait(&bars->v_full[vs], (t / kVSlots) & 1, abort_flag)) break;
          ptx::tc_fence_after();
          const uint32_t vaddr = ptx::smem_addr(sV + vs * C::kTileBytes);
          const uint32_t paddr = tmem + C::kColP + pb * (kBN / 2);  // 16 keys = 8 columns
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint64_t bd = ptx::sdesc_sw128(vaddr + kk * 16 * 128, C::kKVBlock, 1024);
            ptx::mma_bf16_ts(tmem + C::kColO, paddr + kk * 8, bd, idO, (t > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(&bars->v_empty[vs]);
          ptx::mma_commit(&bars->pv_done[pb]);
        }
      }
      ptx::mma_commit(&bars->o_done);
      ptx::mbar_wait(&bars->o_done, 0, abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax rows
    // two threads per row: warps 2-5 take keys [0, 64) of each tile, warps 6-9 keys
    // [64, 128) (warp w and w + 4 read the same TMEM lane quarter); the halves agree on the
    // row max through shared memory and a barrier of the warp pair once per tile
    const int q4 = warp & 3;
    const int h = (warp - 2) >> 2;
    const int r = q4 * 32 + lane;
    const int g = r / a.NT, il = r % a.NT;
    const int node = i0 + il;
    const bool valid = (g < a.G) && (node < a.N) && (r < rows_used);
    const int mnode = valid ? node : 0;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const int c_lo = h * (kBN / 2);  // this thread's key columns in a tile
    const int d_lo = h * (D / 2);    // and its O columns
    const uint32_t pair_bar = 1 + q4;
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory"); };
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    // after a failed wait the loop keeps running without waiting or computing, so that
    // both threads of a row still meet at every pair barrier
    for (int t = 0; t < nt; ++t) {
      const int sb = t & 1;
      if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->s_full[sb], (t >> 1) & 1, abort_flag));
      float sv[kBN / 2];
      if (ok) {
        ptx::tc_fence_after();
        ptx::tmem_ld32(tmem + lane_base + sb * kBN + c_lo, sv);
        ptx::tmem_ld32(tmem + lane_base + sb * kBN + c_lo + 32, sv + 32);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars->s_free[sb]);
      } else {
#pragma unroll
        for (int j = 0; j < kBN / 2; ++j) sv[j] = -INFINITY;
      }

      const int j0 = (t_begin + t) * kBN;
      const uint64_t vis = key_mask(j0 + c_lo, a.P, a.N, mnode, s_par);
      if (vis != ~0ull) {  // tree / tail tiles: hidden keys become -inf (exp -> 0)
#pragma unroll
        for (int j = 0; j < kBN / 2; ++j)
          if (!((vis >> j) & 1ull)) sv[j] = -INFINITY;
      }
      float m8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) m8[k] = sv[k];
#pragma unroll
      for (int j = 8; j < kBN / 2; j += 8)
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = fmaxf(m8[k], sv[j + k]);
      float tm = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      s_xmax[t & 1][h][r] = tm;
      pair_sync();
      tm = fmaxf(tm, s_xmax[t & 1][h ^ 1][r]);
      const float tms = tm * a.c;
      float alpha = 1.f;
      bool need = false;
      if (tms > m_run + kRescaleLog2) {
        if (m_run != -INFINITY) {
          alpha = ptx::ex2(m_run - tms);
          need = true;
        }
        m_run = tms;
      }
      if (__any_sync(0xffffffffu, need) && t > 0 && ok) {
        // O already holds PV(t-1): wait for it, then scale this thread's half of the row
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, abort_flag));
      }
      if (__any_sync(0xffffffffu, need) && t > 0 && ok) {
        ptx::tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
          float ov[32];
          ptx::tmem_ld32(tmem + lane_base + C::kColO + d_lo + c0, ov);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] *= alpha;
          ptx::tmem_st32(tmem + lane_base + C::kColO + d_lo + c0, ov);
        }
        ptx::tmem_wait_st();
      }
      l_run *= alpha;
      // P buffer t & 1 is free once PV(t-2) has completed
      if (t >= 2 && ok)
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->pv_done[sb], ((t >> 1) - 1) & 1, abort_flag));
      if (!ok) continue;  // nothing more to compute or signal for this tile
      // P = 2^(S*c - m_run) on visible keys, bf16 pairs along the key axis, into this
      // thread's 32 columns of the TMEM P buffer (its row's lane)
      float ls8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) ls8[k] = 0.f;
      const bool live = m_run != -INFINITY;
      uint32_t pw[kBN / 4];
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        float pv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          pv[k] = live ? ptx::ex2(fmaf(sv[cc * 8 + k], a.c, -m_run)) : 0.f;
          ls8[k] += pv[k];
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) pw[cc * 4 + k] = ptx::cvt_bf16x2(pv[2 * k], pv[2 * k + 1]);
      }
      l_run += ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
      ptx::tmem_st32u(tmem + lane_base + C::kColP + sb * (kBN / 2) + h * (kBN / 4), pw);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars->p_full[sb]);
    }
    // ---- epilogue: the row's sum is the two halves' sums
    s_xl[h][r] = l_run;
    pair_sync();
    l_run += s_xl[h ^ 1][r];
    bool have_o = false;
    if (nt > 0) {
      ok = ptx::mbar_wait(&bars->o_done, 0, abort_flag) && ok;
      ok = __all_sync(0xffffffffu, ok);
      have_o = ok;
      if (ok) ptx::tc_fence_after();
    }
    const int hh = hk * a.G + g;
    const size_t orow = (((size_t)b * a.Hq + hh) * a.N + node) * D;
    if (a.splits == 1) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        float ov[32];
        if (have_o) {
          ptx::tmem_ld32(tmem + lane_base + C::kColO + d_lo + c0, ov);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] = 0.f;
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + orow + d_lo + c0);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 u;
            u.x = ptx::cvt_bf16x2(ov[8 * k + 0] * inv, ov[8 * k + 1] * inv);
            u.y = ptx::cvt_bf16x2(ov[8 * k + 2] * inv, ov[8 * k + 3] * inv);
            u.z = ptx::cvt_bf16x2(ov[8 * k + 4] * inv, ov[8 * k + 5] * inv);
            u.w = ptx::cvt_bf16x2(ov[8 * k + 6] * inv, ov[8 * k + 7] * inv);
            dst[k] = u;
          }
        }
      }
    } else {
      // park this split's unnormalised O as row-major [128][D] fp32 with the 16-byte chunks
      // of row r XOR-swizzled by (r & 7) (conflict-free 16-byte stores), plus (m, l), in
      // the drained K/V ring for the cluster merge below
      unsigned char* part = sK;
      float2* ml = reinterpret_cast<float2*>(sK + D * kRows * 4);
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        float ov[32];
        if (have_o) {
          ptx::tmem_ld32(tmem + lane_base + C::kColO + d_lo + c0, ov);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int chunk = (d_lo + c0) / 4 + k;
          *reinterpret_cast<float4*>(part + r * D * 4 + ((chunk ^ (r & 7)) << 4)) =
              make_float4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
        }
      }
      if (h == 0) ml[r] = make_float2(have_o ? m_run : -INFINITY, have_o ? l_run : 0.f);
    }
    ptx::tc_fence_before();
  }
  __syncwarp();
  if (a.splits > 1) {
    // The KV splits of this row tile form one thread-block cluster.  After every CTA has
    // parked its partial, CTA `split` merges rows [split*R, split*R + R) by reading all
    // peers' partials through distributed shared memory, then nobody leaves before every
    // peer has finished reading.
    ptx::cluster_sync();
    {
      // every thread; item = (row of this CTA's slice, 16-byte chunk of 4 columns):
      // a warp reads one contiguous row of each peer's partial, all loads issued first
      const int S = a.splits;
      const int R = (kRows + S - 1) / S;
      const int r0 = split * R, r1 = min(kRows, r0 + R);
      const int nrows = max(0, r1 - r0);
      constexpr int kChunks = D / 4;
      const uint32_t part_local = ptx::smem_addr(sK);
      const uint32_t ml_local = ptx::smem_addr(sK + D * kRows * 4);
      for (int item = threadIdx.x; item < nrows * kChunks; item += kThreads) {
        const int rr = r0 + item / kChunks;
        const int ch = item % kChunks;
        const int gg = rr / a.NT, ii = i0 + rr % a.NT;
        if (gg >= a.G || ii >= a.N || rr >= rows_used) continue;
        float2 mlv[kMaxSplits];
        float4 x[kMaxSplits];
        const uint32_t moff = (uint32_t)(rr * 8);
        const uint32_t xoff = (uint32_t)(rr * D * 4 + ((ch ^ (rr & 7)) << 4));
#pragma unroll
        for (int s2 = 0; s2 < kMaxSplits; ++s2) {
          if (s2 < S) {
            mlv[s2] = ptx::ld_cluster_f32x2(ptx::map_cluster(ml_local, s2) + moff);
            x[s2] = ptx::ld_cluster_f32x4(ptx::map_cluster(part_local, s2) + xoff);
          }
        }
        float M = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < kMaxSplits; ++s2)
          if (s2 < S) M = fmaxf(M, mlv[s2].x);
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s2 = 0; s2 < kMaxSplits; ++s2) {
          if (s2 < S && mlv[s2].x != -INFINITY) {
            const float w = ptx::ex2(mlv[s2].x - M);
            L = fmaf(mlv[s2].y, w, L);
            acc.x = fmaf(w, x[s2].x, acc.x);
            acc.y = fmaf(w, x[s2].y, acc.y);
            acc.z = fmaf(w, x[s2].z, acc.z);
            acc.w = fmaf(w, x[s2].w, acc.w);
          }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const size_t o2 = (((size_t)b * a.Hq + hk * a.G + gg) * a.N + ii) * D + ch * 4;
        uint2 u;
        u.x = ptx::cvt_bf16x2(acc.x * inv, acc.y * inv);
        u.y = ptx::cvt_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + o2) = u;
      }
    }
    __syncwarp();
    ptx::cluster_sync();
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && bars->abort) set_dev_status(a.dev_status, TV_DEV_TIMEOUT);
}

// ------------------------------------------------------------------------------------
// host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 3-D bf16 map {D, rows, planes} with a 64 x box_rows x 1 box, 128-byte swizzle.
static bool encode_3d(CUtensorMap* m, const void* base, int D, int rows, long long planes, long long row_stride_elems,
                      long long plane_stride_elems, int box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)row_stride_elems * 2, (cuuint64_t)plane_stride_elems * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

AttnPlan attn_plan(int B, int Hq, int Hkv, int D, int P, int N, tv_dtype dtype) {
  AttnPlan p{};
  const int G = Hkv > 0 ? Hq / Hkv : 0;
  p.tc = dtype == TV_BF16 && (D == 64 || D == 128) && G >= 1 && G <= 16 && (long long)G * N >= 64;
  if (!p.tc) return p;
  p.nt = (kRows / G) / 8 * 8;
  p.mtiles = (N + p.nt - 1) / p.nt;
  p.splits = 1;  // chosen at launch from the device's cluster occupancy
  p.total = 0;   // split partials stay in the cluster's shared memory
  return p;
}

// How many clusters of `s` CTAs of attn_tc_kernel<D> can be resident at once on the
// current device (cached per device, D and s).
template <int D>
static int max_active_clusters(int s) {
  static int cache[64][kMaxSplits + 1];
  static bool init = false;
  if (!init) {
    for (auto& row : cache)
      for (int& v : row) v = -1;
    init = true;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev][s] >= 0) return cache[dev][s];
  using C = TcCfg<D>;
  int n = 0;
  if (cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(s * 64, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemAlloc;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)s;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel<D>, &cfg) != cudaSuccess) n = 0;
  }
  cache[dev][s] = n;
  return n;
}

// KV splits per row tile: minimise (waves of clusters) x (KV tiles per CTA + a fixed
// per-CTA cost for set-up and the cluster merge), counted in 64-key tiles.
template <int D>
static int choose_splits(long long row_tiles, int t_all) {
  constexpr double kFixedTiles = 1.5;
  // with an SM share set for concurrent kernels, plan for that part of the device
  const int share = sm_share_attention();
  int nsm = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  int best = 1;
  double best_cost = 1e300;
  for (int s = 1; s <= kMaxSplits && s <= t_all; ++s) {
    int act = max_active_clusters<D>(s);
    if (act <= 0) continue;
    if (share > 0 && share < nsm) act = std::max(1, (int)((long long)act * share / nsm));
    const long long waves = (row_tiles + act - 1) / act;
    const double cost = (double)waves * ((t_all + s - 1) / s + kFixedTiles);
    if (cost < best_cost * 0.98) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

template <int D>
static cudaError_t launch_tc_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const TcArgs& a,
                               int B, int Hkv, cudaStream_t stream) {
  using C = TcCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.MT * a.splits, Hkv, B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<D>, mq, mk, mv, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attn_tc(const void* q, const void* k, const void* v, void* out, const int32_t* parent, int B,
                           int Hq, int Hkv, int D, int P, int N, int S, float scale, const AttnPlan& plan, char* ws,
                           int32_t* dev_status, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!encode_3d(&mq, q, D, N, (long long)B * Hq, D, (long long)N * D, plan.nt)) return cudaErrorInvalidValue;
  if (!encode_3d(&mk, k, D, P + N, (long long)B * Hkv, D, (long long)S * D, kBN)) return cudaErrorInvalidValue;
  if (!encode_3d(&mv, v, D, P + N, (long long)B * Hkv, D, (long long)S * D, kBN)) return cudaErrorInvalidValue;
  TcArgs a;
  a.out = out;
  a.parent = parent;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.N = N;
  a.P = P;
  a.G = Hq / Hkv;
  a.NT = plan.nt;
  a.MT = plan.mtiles;
  a.c = scale * kLog2e;
  a.dev_status = dev_status;
  const long long row_tiles = (long long)B * Hkv * plan.mtiles;
  const int t_all = (P + N + kBN - 1) / kBN;
  a.splits = D == 64 ? choose_splits<64>(row_tiles, t_all) : choose_splits<128>(row_tiles, t_all);
  if (D == 64) return launch_tc_d<64>(mq, mk, mv, a, B, Hkv, stream);
  return launch_tc_d<128>(mq, mk, mv, a, B, Hkv, stream);
}

}  // namespace tv
