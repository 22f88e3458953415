// dQ of the recompute backward as a separate pass with no atomics, so that
// dQ is the same bit for bit on every run (the summary's backward,
// "Recomputation", leaves the order of the dQ sum open; this pass fixes it).
// One CTA owns one query tile i of one (batch, head) and walks the key tiles
// j that reach it in ascending order:
//   S = Q_i K_j^T,  P = exp(scale*S - lse_i),  dP = dO_i V_j^T,
//   dS = P o (dP - D_i),  dQ_i += dS K_j,
// then writes bf16(scale * dQ_i) straight from the accumulator.  Each dQ
// element is one CTA's fixed-order sum, so no fp32 workspace and no
// conversion pass are needed.  The key-tile pass (fa_bwd_kernel without its
// dQ product) supplies dK and dV, which it already sums in a fixed order.
//
// GB300 design (one CTA = one head x one 128-row query tile):
//   warp 0      TMA producer: Q_i, dO_i once; K_j, V_j through an NS-stage ring
//   warp 1      allocates 512 TMEM columns; lane 0 issues the MMAs
//   warps 4-11  one thread per query row and half of the key columns (warps
//               4-7: keys 0-63, warps 8-11: keys 64-127): P from S and lse,
//               dS from dP and D into shared memory (bf16, 128-byte swizzle);
//               at the end the dQ accumulator to global memory
//   warps 2-3   idle
// TMEM: S [0,128), dP [128,256), dQ [256, 256+d).
// The dS buffer is single: dP of tile j+1 is issued after dQ of tile j, and
// a commit tracks every earlier MMA of the issuing thread, so dP(j+1) having
// completed means dQ(j) has finished reading dS(j).
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_sched.cuh"

namespace fa {
namespace {

template <int D>
struct DqSmem {
  static constexpr int CH = D / 64;
  static constexpr int CHUNK = kTile * 128;  // 128 rows x 64 bf16
  static constexpr int TILE = CH * CHUNK;
  static constexpr int NS = (D == 64) ? 3 : 2;  // K/V stages
  static constexpr int Q = 0;
  static constexpr int DO = Q + TILE;
  static constexpr int KV = DO + TILE;  // stage s: K at KV + 2 s TILE, V after it
  static constexpr int DS = KV + NS * 2 * TILE;
  static constexpr int BAR = DS + 2 * CHUNK;
  static constexpr int B_QDO = 0, B_KVF = 1, B_KVE = B_KVF + NS, B_SF = B_KVE + NS,
                       B_DPF = B_SF + 1, B_PR = B_DPF + 1, B_DSR = B_PR + 1, B_FIN = B_DSR + 1,
                       NBAR = B_FIN + 1;
  static constexpr int MISC = BAR + NBAR * 8;
  static constexpr int ALLOC = MISC + 16 + 1024;
  static_assert(ALLOC <= 232448, "shared memory budget");
  static constexpr int T_S = 0, T_DP = 128, T_DQ = 256;
};

constexpr int kDqThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
__global__ void __launch_bounds__(kDqThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv,
                     const __grid_constant__ CUtensorMap tdo, const DqParams p) {
  using L = DqSmem<D>;
  grid_dep_wait();  // the previous kernel's writes are visible from here on
  grid_dep_launch();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) { return sb + L::BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N;
  const int nT = (N + kTile - 1) / kTile;
  const int BH = p.B * p.H;
  int bh, qt;
  fwd_cta_coords(blockIdx.x, BH, nT, p.causal != 0, bh, qt);  // causal: longest rows first
  const int head = bh % p.H;

  // key tiles of query tile qt: 0 .. qt (causal), all, or its CSR list
  FwdSchedule sch;
  sch.init(qt, nT, p.causal != 0, p.lists, head, true);

  // Thread 0 (the producer's lane) initialises the barriers and sends Q, dO
  // and the first K/V pair at once, before the block-wide barrier and the
  // TMEM allocation.
  bool pre_kv = false;  // thread 0: the first key tile's K and V are in flight
  if (threadIdx.x == 0) {
    mbar_init(bar(L::B_QDO), 1);
    for (int s = 0; s < L::NS; ++s) {
      mbar_init(bar(L::B_KVF + s), 1);
      mbar_init(bar(L::B_KVE + s), 1);
    }
    mbar_init(bar(L::B_SF), 1);
    mbar_init(bar(L::B_DPF), 1);
    mbar_init(bar(L::B_PR), 256);
    mbar_init(bar(L::B_DSR), 256);
    mbar_init(bar(L::B_FIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    prefetch_tmap(&tdo);
    mbar_arrive_expect_tx(bar(L::B_QDO), 2 * L::TILE);
#pragma unroll
    for (int c = 0; c < L::CH; ++c) {
      tma_load_3d(sb + L::Q + c * L::CHUNK, &tq, bar(L::B_QDO), 64 * c, qt * kTile, bh);
      tma_load_3d(sb + L::DO + c * L::CHUNK, &tdo, bar(L::B_QDO), 64 * c, qt * kTile, bh);
    }
    FwdSchedule first = sch;  // the first key tile, without advancing sch
    int kt0, mem0;
    if (first.next(kt0, mem0)) {  // ring slot 0
      mbar_arrive_expect_tx(bar(L::B_KVF), 2 * L::TILE);
#pragma unroll
      for (int c = 0; c < L::CH; ++c) {
        tma_load_3d(sb + L::KV + c * L::CHUNK, &tk, bar(L::B_KVF), 64 * c, kt0 * kTile, bh);
        tma_load_3d(sb + L::KV + L::TILE + c * L::CHUNK, &tv, bar(L::B_KVF), 64 * c,
                    kt0 * kTile, bh);
      }
      pre_kv = true;
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, p.err, p.wait_ns};

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      // Q, dO and the first K/V pair went out before the block-wide barrier
      uint32_t idx = pre_kv ? 1 : 0;
      bool ok = true;
      bool skip = pre_kv;
      int kt, mem;
      while (ok && sch.next(kt, mem)) {
        if (skip) {
          skip = false;
          continue;
        }
        const int pos = idx % L::NS;
        const uint32_t round = idx / L::NS;
        if (round > 0 && !wait_bar(bar(L::B_KVE + pos), (round - 1) & 1, wc)) {
          ok = false;
          break;
        }
        const uint32_t kdst = sb + L::KV + pos * 2 * L::TILE;
        mbar_arrive_expect_tx(bar(L::B_KVF + pos), 2 * L::TILE);
#pragma unroll
        for (int c = 0; c < L::CH; ++c) {
          tma_load_3d(kdst + c * L::CHUNK, &tk, bar(L::B_KVF + pos), 64 * c, kt * kTile, bh);
          tma_load_3d(kdst + L::TILE + c * L::CHUNK, &tv, bar(L::B_KVF + pos), 64 * c,
                      kt * kTile, bh);
        }
        ++idx;
      }
      // let copies still in flight land before the CTA can exit
      drain_bar(bar(L::B_QDO), 0, p.wait_ns);
      if (!ok) {
        const uint32_t first = idx > static_cast<uint32_t>(L::NS) ? idx - L::NS : 0;
        for (uint32_t j = first; j < idx; ++j)
          drain_bar(bar(L::B_KVF + j % L::NS), (j / L::NS) & 1, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);  // S, dP
      constexpr uint32_t idDQ = idesc_bf16(128, D, false, true);     // dQ
      // X[128 q x 128 k] = A[128 x D] B[128 x D]^T, both K-major
      // operand descriptors formed once and advanced per k-step
      const uint64_t dk0 = desc_sw128(sb, 16, 1024), dm0 = desc_sw128(sb, L::CHUNK, 1024);
      auto issue_qk = [&](uint32_t dst, uint32_t a, uint32_t b) {
        const uint64_t da = desc_advance(dk0, a - sb), db = desc_advance(dk0, b - sb);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::CHUNK + (kk & 3) * 32;
          mma_bf16_ss(dst, desc_advance(da, off), desc_advance(db, off), idSS, kk > 0);
        }
      };
      // dQ[128 q x D] += dS[128 q x 128 k] K[128 k x D] (K is MN-major here)
      auto issue_dq = [&](uint32_t dst, uint32_t kaddr, bool acc) {
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * L::CHUNK + (kk & 3) * 32;
          mma_bf16_ss(dst, desc_advance(dk0, L::DS + aoff), desc_advance(dm0, kaddr - sb + kk * 2048),
                      idDQ, (acc || kk > 0) ? 1u : 0u);
        }
      };
      const uint32_t tS = tmem + L::T_S, tDP = tmem + L::T_DP, tDQ = tmem + L::T_DQ;
      auto kv_addr = [&](uint32_t idx) { return sb + L::KV + (idx % L::NS) * 2 * L::TILE; };
      int kt, mem;
      bool ok = wait_bar(bar(L::B_QDO), 0, wc);
      bool have = sch.next(kt, mem);
      uint32_t n = 0;
      if (ok && have) {
        ok = wait_bar(bar(L::B_KVF + 0), 0, wc);
        if (ok) {
          tc_fence_after();
          issue_qk(tS, sb + L::Q, kv_addr(0));
          mma_commit(bar(L::B_SF));
          issue_qk(tDP, sb + L::DO, kv_addr(0) + L::TILE);
          mma_commit(bar(L::B_DPF));
        }
      }
      while (ok && have) {
        const bool have_n = sch.next(kt, mem);
        const uint32_t n1 = n + 1;
        // S of the next tile once P has been read out of the S columns
        if (!(ok = wait_bar(bar(L::B_PR), n & 1, wc))) break;
        if (have_n) {
          if (!(ok = wait_bar(bar(L::B_KVF + n1 % L::NS), (n1 / L::NS) & 1, wc))) break;
          tc_fence_after();
          issue_qk(tS, sb + L::Q, kv_addr(n1));
          mma_commit(bar(L::B_SF));
        }
        // dQ += dS K_j once dS is in shared memory; then K_j, V_j are free
        if (!(ok = wait_bar(bar(L::B_DSR), n & 1, wc))) break;
        tc_fence_after();
        issue_dq(tDQ, kv_addr(n), n > 0);
        mma_commit(bar(L::B_KVE + n % L::NS));
        if (have_n) {
          issue_qk(tDP, sb + L::DO, kv_addr(n1) + L::TILE);
          mma_commit(bar(L::B_DPF));
        }
        have = have_n;
        n = n1;
      }
      mma_commit(bar(L::B_FIN));
      drain_bar(bar(L::B_FIN), 0, p.wait_ns);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------ P, dS warps
    const int half = (warp - 4) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_off + L::T_S + 64 * half;
    const uint32_t tDP = tmem + lane_off + L::T_DP + 64 * half;
    const uint32_t tDQ = tmem + lane_off + L::T_DQ + (D / 2) * half;
    const uint32_t dsbuf = sb + L::DS + half * L::CHUNK;
    const float sl2 = p.scale * kLog2e;
    const int qrow = qt * kTile + r;
    const size_t row_idx = static_cast<size_t>(bh) * N + (qrow < N ? qrow : 0);
    const float lse_c = p.lse[row_idx];
    const float dlt_c = p.delta[row_idx];
    const bool live = qrow < N && lse_c != -INFINITY;
    const float lse2 = live ? lse_c * kLog2e : 0.f;
    const uint64_t sl2x2 = f2_pack(sl2, sl2), nlse2x2 = f2_pack(-lse2, -lse2);
    const uint64_t dltx2 = f2_pack(dlt_c, dlt_c);
    bool ok = true;
    uint32_t n = 0;
    int kt, mem;
    while (ok && sch.next(kt, mem)) {
      ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_SF), n & 1, wc));
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[2][32];
      tmem_ld32(tS, sv[0]);
      tmem_ld32(tS + 32, sv[1]);
      tmem_ld_wait();
      reg_fence(sv[0]);
      reg_fence(sv[1]);
      const int kcol0 = kt * kTile + 64 * half;  // first key of this thread's columns
      const bool need_mask = (kcol0 + 64 > N) || (p.causal && kcol0 + 63 > qt * kTile);
      // keys kcol0 + i with i >= lim are masked (past N, or after this row
      // when causal)
      int lim = N - kcol0;
      if (p.causal && qrow - kcol0 + 1 < lim) lim = qrow - kcol0 + 1;
      uint32_t pw[32];  // pw[i]: keys 2i, 2i+1 of this thread's 64 columns
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        // exponent arguments of two keys in one fp32 x2 FMA
        float a, b;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[i >> 4][(2 * i) & 31]),
                                 __uint_as_float(sv[i >> 4][(2 * i + 1) & 31])),
                         sl2x2, nlse2x2),
                  a, b);
        a = ex2(a);
        b = ex2(b);
        if (need_mask) {
          if (2 * i >= lim) a = 0.f;
          if (2 * i + 1 >= lim) b = 0.f;
        }
        pw[i] = live ? pack_bf16(a, b) : 0u;
      }
      tc_fence_before();
      mbar_arrive(bar(L::B_PR));
      // dS = P o (dP - D_i)
      ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_DPF), n & 1, wc));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t dp[32];
        tmem_ld32(tDP + 32 * c, dp);
        tmem_ld_wait();
        reg_fence(dp);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t pp = pw[16 * c + 4 * g + j];
            // P o (dP - D) for two keys in fp32 x2
            float x0, x1;
            f2_unpack(f2_mul(f2_pack(bf16_lo(pp), bf16_hi(pp)),
                             f2_sub(f2_pack(__uint_as_float(dp[8 * g + 2 * j]),
                                            __uint_as_float(dp[8 * g + 2 * j + 1])),
                                    dltx2)),
                      x0, x1);
            w[j] = pack_bf16(x0, x1);
          }
          st_shared_v4(dsbuf + sw128_offset(r, 4 * c + g), w[0], w[1], w[2], w[3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(L::B_DSR));
      ++n;
    }
    // ---------------------------------------------------- epilogue: dQ
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_FIN), 0, wc));
    tc_fence_after();
    if (ok) {  // warp-uniform: every lane takes part in the TMEM reads
      // This thread's D/2 columns of its row are packed into the Q tile (no
      // MMA reads it any more), in the row's half of the 128-byte-swizzled
      // layout; then each store writes whole row pieces of 32 rows.
      constexpr int U = D / 16;  // 16-byte units per thread row (D/2 bf16)
      const uint32_t qbuf = sb + L::Q + (D == 128 ? half * L::CHUNK : 0);
      const int u0 = (D == 64) ? 4 * half : 0;  // first unit of this half in the row
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t a[32];
        if (n > 0) {
          tmem_ld32(tDQ + 32 * c, a);
          tmem_ld_wait();
          reg_fence(a);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) a[j] = 0u;
        }
#pragma unroll
        for (int v = 0; v < 4; ++v)
          st_shared_v4(qbuf + sw128_offset(r, u0 + 4 * c + v),
                       pack_bf16(__uint_as_float(a[8 * v + 0]) * p.scale,
                                 __uint_as_float(a[8 * v + 1]) * p.scale),
                       pack_bf16(__uint_as_float(a[8 * v + 2]) * p.scale,
                                 __uint_as_float(a[8 * v + 3]) * p.scale),
                       pack_bf16(__uint_as_float(a[8 * v + 4]) * p.scale,
                                 __uint_as_float(a[8 * v + 5]) * p.scale),
                       pack_bf16(__uint_as_float(a[8 * v + 6]) * p.scale,
                                 __uint_as_float(a[8 * v + 7]) * p.scale));
      }
      __syncwarp();
      const int qrow0 = qt * kTile + q4 * 32;  // this warp's first row
      uint8_t* dst = static_cast<uint8_t*>(p.dq) +
                     ((static_cast<size_t>(bh) * N + qrow0) * D + (D / 2) * half) * 2;
      constexpr int RPI = 32 / U;  // rows per store instruction
#pragma unroll
      for (int it = 0; it < 32 / RPI; ++it) {
        const int j = it * RPI + lane / U, v = lane % U;
        const uint4 w = ld_shared_v4(qbuf + sw128_offset(q4 * 32 + j, u0 + v));
        if (qrow0 + j < N)
          *reinterpret_cast<uint4*>(dst + static_cast<size_t>(j) * D * 2 + v * 16) = w;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_dq_d(const DqParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const CUtensorMap& tdo, cudaStream_t stream) {
  using L = DqSmem<D>;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e =
      smem_attr_once(attr_done, reinterpret_cast<const void*>(fa_bwd_dq_kernel<D>), L::ALLOC);
  if (e != cudaSuccess) return e;
  const int nT = (p.N + kTile - 1) / kTile;
  const long long ctas = static_cast<long long>(nT) * p.B * p.H;
  return launch_pdl(fa_bwd_dq_kernel<D>, dim3(static_cast<unsigned>(ctas)), dim3(kDqThreads),
                    L::ALLOC, stream, tq, tk, tv, tdo, p);
}

}  // namespace

cudaError_t launch_backward_dq(const DqParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv, const CUtensorMap& tdo,
                               cudaStream_t stream) {
  if (p.d == 64) return launch_dq_d<64>(p, tq, tk, tv, tdo, stream);
  if (p.d == 128) return launch_dq_d<128>(p, tq, tk, tv, tdo, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
