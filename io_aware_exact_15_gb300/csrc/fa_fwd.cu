// Forward pass of exact attention, tile by tile with an online softmax
// (FlashAttention hackmd summary, "Tiling" and "Kernel Fusion": Q, K, V are
// split into blocks that are brought on chip, the row max m and the row sum
// l of exponentials are carried from block to block, and O is rescaled so
// the final result equals the full softmax; one kernel does
// matmul -> mask -> softmax -> matmul and only O and the statistics reach
// HBM).  The statistic written is lse = m + ln l.
//
// GB300 design (one CTA = one head x two 128-row query tiles):
//   warp 0      TMA producer: both Q tiles once, then K_j, V_j through an
//               NS-deep ring of 128 x d tiles (128-byte swizzle)
//   warp 1      allocates 512 TMEM columns; an elected lane issues every
//               tcgen05.mma (the whole warp runs the issue loop):
//               S_s = Q_s K_j^T (fp32 in TMEM) and O_s += P_s V_j
//   warps 2-5   softmax for query tile 0, warps 6-9 for query tile 1: one
//               thread per query row reads its 128 scores from TMEM, applies
//               the causal / ragged-length mask, updates (m, l) in the log2
//               domain with the scale folded into one FMA before ex2, writes
//               P (bf16) back into TMEM over the scores it has read (the PV
//               MMA takes its A operand from TMEM), and rescales its
//               O row in TMEM only when the running max grew by more than
//               2^8 (the final O / l uses the same m, so this stays exact).
// While one warpgroup does its softmax the tensor core runs the other tile's
// MMAs.  TMEM columns: S0 [0,128) S1 [128,256) O0 [256,256+d) O1 [.., +d);
// P_s takes the first 64 columns of S_s and the MMA issuer puts PV_s(j)
// before S_s(j+1) in its stream: the tensor core runs one CTA's MMAs in
// issue order, so P_s is read before the next scores overwrite it.  The K/V
// ring is 5 (d = 128) or 8 (d = 64) tiles.
//
// Compact form (grids of at most four waves of two-tile CTAs, and every
// grid with a block mask): one query
// tile per CTA, warps 0-5 only, 256 TMEM columns (S [0,128), O [128,128+d)),
// a 2 (d = 128) or 4 (d = 64) tile ring, so that two CTAs share an SM.  The
// block-size sweep also builds key tiles of 64 and 256 keys (template BC).
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_philox.cuh"
#include "fa_sched.cuh"

namespace fa {
namespace {

// BC: keys per key tile (128 except in the block-size sweep: 64 or 256).
// CMP: the compact form of a one-query-tile CTA: 6 warps, tensor memory and
// shared memory sized for one tile, so that two CTAs can share an SM where
// both fit (at most 256 TMEM columns and ~113 KB of shared memory each).
template <int D, int NS_ = 0, int BC = kTile, bool CMP = false>
struct FwdSmem {
  static constexpr int CH = D / 64;             // 128-byte column chunks per row
  static constexpr int CHUNK = kTile * 128;     // query tile: [128 rows x 128 B] = 16 KB
  static constexpr int TILE = CH * CHUNK;       // one 128 x D bf16 query tile
  static constexpr int KCHUNK = BC * 128;       // key / value tile: [BC rows x 128 B]
  static constexpr int KTILE = CH * KCHUNK;     // one BC x D bf16 key or value tile
  static constexpr int KBOX = BC < kTile ? BC : kTile;  // rows of one K/V TMA box
  // query tiles per CTA in tensor memory (S and O of each: BC + D columns)
  static constexpr int NQT = CMP ? 1 : 2;
  static_assert(NQT * (BC + D) <= 512, "tensor memory budget");
  static constexpr int QT = CMP ? 1 : 2;  // query tiles in shared memory
  static constexpr int THREADS = CMP ? 192 : 320;
  // columns allocated: the power of two that holds S and O of every tile
  static constexpr int TCOLS = CMP ? (NQT * (BC + D) <= 128   ? 128
                                      : NQT * (BC + D) <= 256 ? 256
                                                              : 512)
                                   : 512;
  // K/V ring slots (one tile each); NS_ != 0 overrides for the tile sweep.
  // The compact form keeps its shared memory within half an SM's.
  static constexpr int NS = NS_ != 0 ? NS_ : CMP ? ((D == 64) ? 4 : 2) : ((D == 64) ? 8 : 5);
  static constexpr int Q = 0;
  static constexpr int KV = Q + QT * TILE;
  static constexpr int BAR = KV + NS * KTILE;
  static constexpr int B_Q = 0, B_KVF = 1, B_KVE = 1 + NS, B_SF = 1 + 2 * NS, B_PF = B_SF + 2,
                       B_OF = B_PF + 2, NBAR = B_OF + 1;
  static constexpr int MISC = BAR + NBAR * 8;
  // TMEM columns of P_s: the first 64 columns of S_s (already read into
  // registers).  d = 64 would leave room for separate P columns after O1,
  // but that layout measured 8 % slower on the BERT-shaped workload.
  static constexpr int T_P = 0;
  static constexpr int T_PSTRIDE = BC;
  static constexpr int T_O = NQT * BC;  // O_s at T_O + s * D
  static constexpr int ALLOC = MISC + 16 + 1024;  // + slack for 1024-byte alignment
  static_assert(ALLOC <= 232448, "shared memory budget");
  // CTAs per SM the launch bounds ask for (registers then capped at 168)
  static constexpr int MINB = (CMP && TCOLS <= 256 && ALLOC <= 113 * 1024) ? 2 : 1;
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (factor 256)

template <int D, int KIND, int NS_, int BC, bool CMP>
__global__ void __launch_bounds__(FwdSmem<D, NS_, BC, CMP>::THREADS,
                                  FwdSmem<D, NS_, BC, CMP>::MINB)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  using L = FwdSmem<D, NS_, BC, CMP>;
  static_assert(BC == kTile || (NS_ != 0 && KIND == kPlain),
                "key tiles other than 128 exist only in the plain sweep instantiations");
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
  // one query tile per CTA: the compact instantiations
  constexpr bool single = L::NQT == 1;
  const int ntmax = (p.N + kTile - 1) / kTile;
  const int npairs = single ? ntmax : (ntmax + 1) / 2;
  const int BH = p.B * p.H;
  int bh, pair;
  fwd_cta_coords(blockIdx.x, BH, npairs, p.causal != 0, bh, pair);
  const int head = bh % p.H;
  // Sequence geometry: length N, first row row0 of the sequence in its
  // slice, the TMA slices zq (Q, O) and zkv (K, V).  Grouped K/V has H / Hkv
  // query heads per key/value head: bh / (H / Hkv) = b * Hkv + h / (H / Hkv).
  // The plain instantiation carries no index arithmetic at all.
  constexpr bool DROP = KIND == kGeneralDropout;
  int N = p.N, row0 = 0, zq = bh, zkv = bh;
  if (KIND == kGrouped || KIND >= kGeneral) zkv = bh / (p.H / p.Hkv);
  const bool varlen = KIND >= kGeneral && p.cu_seqlens != nullptr;
  if (varlen) {
    // variable-length batch: slices are heads, sequences are row ranges
    // (indices clamped to [0, total], so bad offsets cannot write outside)
    const int b = bh / p.H;
    const int a = min(max(p.cu_seqlens[b], 0), p.total);
    const int e = min(max(p.cu_seqlens[b + 1], a), p.total);
    row0 = a;
    N = min(e - a, p.N);
    zq = head;
    zkv = head / (p.H / p.Hkv);
    if ((single ? pair : 2 * pair) * kTile >= N) return;  // no query tile here (CTA-uniform)
  }
  const size_t slice_rows = varlen ? static_cast<size_t>(p.total) : static_cast<size_t>(p.N);
  const int nT = (N + kTile - 1) / kTile;

  FwdScheduleT<BC> sch;
  sch.init(pair, nT, p.causal != 0, p.lists, head, single, (N + BC - 1) / BC);
  // K_j or V_j into ring slot `pos`: CH column chunks of BC / KBOX boxes
  auto load_kv = [&](int pos, const CUtensorMap* m, int kt) {
#pragma unroll
    for (int c = 0; c < L::CH; ++c)
#pragma unroll
      for (int h = 0; h < BC / L::KBOX; ++h)
        tma_load_3d(sb + L::KV + pos * L::KTILE + c * L::KCHUNK + h * L::KBOX * 128, m,
                    bar(L::B_KVF + pos), 64 * c, row0 + kt * BC + h * L::KBOX, zkv);
  };

  // Thread 0 (the producer's lane) initialises the barriers and sends Q and
  // the first K/V pair at once, before the block-wide barrier and the TMEM
  // allocation, so that the first loads start as early as they can.
  bool pre_kv = false;  // thread 0: the first key tile's K and V are in flight
  if (threadIdx.x == 0) {
    mbar_init(bar(L::B_Q), 1);
    for (int s = 0; s < L::NS; ++s) {
      mbar_init(bar(L::B_KVF + s), 1);
      mbar_init(bar(L::B_KVE + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::B_SF + s), 1);
      mbar_init(bar(L::B_PF + s), 128);
    }
    mbar_init(bar(L::B_OF), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    const int y0 = sch.qt[0] * kTile;
    const int y1 = (sch.act[1] ? sch.qt[1] : sch.qt[0]) * kTile;
    mbar_arrive_expect_tx(bar(L::B_Q), L::QT * L::TILE);
#pragma unroll
    for (int c = 0; c < L::CH; ++c) {
      tma_load_3d(sb + L::Q + c * L::CHUNK, &tq, bar(L::B_Q), 64 * c, row0 + y0, zq);
      if (L::QT == 2)
        tma_load_3d(sb + L::Q + L::TILE + c * L::CHUNK, &tq, bar(L::B_Q), 64 * c, row0 + y1, zq);
    }
    FwdScheduleT<BC> first = sch;  // the first key tile, without advancing sch
    int kt0, mem0;
    if (first.next(kt0, mem0)) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {  // ring slots 0 and 1
        mbar_arrive_expect_tx(bar(L::B_KVF + t), L::KTILE);
        load_kv(t, t == 0 ? &tk : &tv, kt0);
      }
      pre_kv = true;
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::TCOLS);
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
      // Q and the first K/V pair went out before the block-wide barrier
      uint32_t idx = pre_kv ? 2 : 0;
      bool ok = true;
      bool skip = pre_kv;
      int kt, mem;
      while (ok && sch.next(kt, mem)) {
        if (skip) {
          skip = false;
          continue;
        }
        for (int t = 0; t < 2; ++t) {
          const int pos = idx % L::NS;
          const uint32_t round = idx / L::NS;
          if (round > 0 && !wait_bar(bar(L::B_KVE + pos), (round - 1) & 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(L::B_KVF + pos), L::KTILE);
          load_kv(pos, t == 0 ? &tk : &tv, kt);
          ++idx;
        }
      }
      // let copies still in flight land before the CTA can exit
      drain_bar(bar(L::B_Q), 0, p.wait_ns);
      if (!ok) {
        const uint32_t first = idx > static_cast<uint32_t>(L::NS) ? idx - L::NS : 0;
        for (uint32_t j = first; j < idx; ++j)
          drain_bar(bar(L::B_KVF + j % L::NS), (j / L::NS) & 1, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    // The whole warp runs the issuer (waits and tests are warp votes, so
    // control flow and operand descriptors are warp-uniform) and the
    // elected lane issues each MMA and commit.
    {
      auto uwait = [&](uint32_t b, uint32_t ph) {
        return __all_sync(0xffffffffu, wait_bar(b, ph, wc));
      };
      auto utry = [&](uint32_t b, uint32_t ph) { return __all_sync(0xffffffffu, mbar_try(b, ph)); };
      auto ecommit = [&](uint32_t b) {
        if (elect_one()) mma_commit(b);
      };
      constexpr uint32_t idS = idesc_bf16(128, BC, false, false);
      constexpr uint32_t idO = idesc_bf16(128, D, false, true);
      // descriptors are formed once per operand and advanced per k-step
      const uint64_t dq0 = desc_sw128(sb + L::Q, 16, 1024);
      const uint64_t dkv0 = desc_sw128(sb + L::KV, 16, 1024);  // K-major ring slot 0
      const uint64_t dv0 = desc_sw128(sb + L::KV, L::KCHUNK, 1024);  // MN-major ring slot 0
      auto issue_s = [&](int s, int kpos) {
        const uint64_t qa = desc_advance(dq0, s * L::TILE);
        const uint64_t kb = desc_advance(dkv0, kpos * L::KTILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t in_row = (kk & 3) * 32;
          const uint64_t da = desc_advance(qa, (kk >> 2) * L::CHUNK + in_row);
          const uint64_t db = desc_advance(kb, (kk >> 2) * L::KCHUNK + in_row);
          if (elect_one()) mma_bf16_ss(tmem + s * BC, da, db, idS, kk > 0);
        }
      };
      // O_s += P_s V: P_s sits in TMEM (BC / 2 columns, two bf16 per column),
      // V is MN-major in shared memory
      auto issue_pv = [&](int s, int vpos, bool acc) {
        const uint64_t vb = desc_advance(dv0, vpos * L::KTILE);
#pragma unroll
        for (int kk = 0; kk < BC / 16; ++kk) {
          const uint64_t db = desc_advance(vb, kk * 2048);
          if (elect_one())
            mma_bf16_ts(tmem + L::T_O + s * D, tmem + L::T_P + s * L::T_PSTRIDE + kk * 8, db, idO,
                        (acc || kk > 0) ? 1u : 0u);
        }
      };
      int kt, mem, kt_n = 0, mem_n = 0;
      uint32_t idx = 0;
      uint32_t cnt01 = 0;  // participations of slot 0 (low 16 bits) and slot 1 (high)
      bool ok = uwait(bar(L::B_Q), 0);
      bool have = sch.next(kt, mem);
      if (ok && have) {
        const int kpos = idx % L::NS;
        ok = uwait(bar(L::B_KVF + kpos), (idx / L::NS) & 1);
        if (ok) {
          tc_fence_after();
          for (int s = 0; s < 2; ++s)
            if (mem & (1 << s)) {
              issue_s(s, kpos);
              ecommit(bar(L::B_SF + s));
            }
          ecommit(bar(L::B_KVE + kpos));
          ++idx;
        }
      }
      while (ok && have) {
        const bool have_n = sch.next(kt_n, mem_n);
        const int vpos = idx % L::NS;
        ok = uwait(bar(L::B_KVF + vpos), (idx / L::NS) & 1);
        ++idx;
        if (!ok) break;
        tc_fence_after();
        int kpos = -1;
        for (int s = 0; s < 2 && ok; ++s) {
          if (mem & (1 << s)) {
            const uint32_t cs = (cnt01 >> (16 * s)) & 0xFFFFu;
            ok = uwait(bar(L::B_PF + s), cs & 1);
            if (!ok) break;
            tc_fence_after();
            issue_pv(s, vpos, cs > 0);
            cnt01 += 1u << (16 * s);
          }
          if (have_n && (mem_n & (1 << s))) {
            if (kpos < 0) {
              kpos = idx % L::NS;
              ok = uwait(bar(L::B_KVF + kpos), (idx / L::NS) & 1);
              if (!ok) break;
              tc_fence_after();
            }
            issue_s(s, kpos);
            ecommit(bar(L::B_SF + s));
          }
        }
        if (!ok) break;
        ecommit(bar(L::B_KVE + vpos));
        if (kpos >= 0) {
          ecommit(bar(L::B_KVE + kpos));
          ++idx;
        }
        kt = kt_n;
        mem = mem_n;
        have = have_n;
      }
      // every MMA issued above completes before o_full fires
      ecommit(bar(L::B_OF));
      drain_bar(bar(L::B_OF), 0, p.wait_ns);
    }
  } else {
    // ------------------------------------------------------ softmax warps
    const int s = (warp - 2) >> 2;
    const int q4 = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q4 * 32 + lane;
    const int qt = sch.qt[s];
    const bool active = sch.act[s];
    const int qrow = qt * kTile + r;
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_off + s * BC;
    const uint32_t tO = tmem + lane_off + L::T_O + s * D;
    const uint32_t tP = tmem + lane_off + L::T_P + s * L::T_PSTRIDE;
    const float sl2 = p.scale * kLog2e;
    const DropoutRng rng{p.drop.rk, p.drop.offset, p.drop.t * 0x01010101u};
    float m = -INFINITY, l = 0.f;
    int cnt = 0;
    bool ok = true;
    int kt, mem;
    while (ok && sch.next(kt, mem)) {
      if (!(mem & (1 << s))) continue;
      ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_SF + s), cnt & 1, wc));
      if (!ok) break;
      tc_fence_after();
      // The scores of a key tile are read in register groups of up to 128
      // keys (GC chunks of 32); a 256-key tile (block-size sweep) takes two
      // groups, read once for the row max and again for the exponentials.
      constexpr int GW = BC < kTile ? BC : kTile;
      constexpr int NG = BC / GW;
      constexpr int GC = GW / 32;
      const int kbase = kt * BC;
      const bool need_mask = (kbase + BC > N) || (p.causal && kbase + BC - 1 > qt * kTile);
      uint32_t sr[GC][32];
      auto load_group = [&](int g) {
#pragma unroll
        for (int c = 0; c < GC; ++c) tmem_ld32(tS + g * GW + 32 * c, sr[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < GC; ++c) reg_fence(sr[c]);
        if (need_mask) {
          // keys kbase + i with i >= lim are masked (past N, or after this
          // row when causal)
          int lim = N - kbase;
          if (p.causal && qrow - kbase + 1 < lim) lim = qrow - kbase + 1;
#pragma unroll
          for (int c = 0; c < GC; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (g * GW + 32 * c + j >= lim) sr[c][j] = __float_as_uint(-INFINITY);
        }
      };
      float mx[GC];
#pragma unroll
      for (int c = 0; c < GC; ++c) mx[c] = -INFINITY;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        load_group(g);
#pragma unroll
        for (int j = 0; j < 32; j += 2)  // two scores per three-input max
#pragma unroll
          for (int c = 0; c < GC; ++c)
            mx[c] = fmax3(mx[c], __uint_as_float(sr[c][j]), __uint_as_float(sr[c][j + 1]));
      }
      float mxa;
      if constexpr (GC == 4) {
        mxa = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      } else {
        mxa = mx[0];
#pragma unroll
        for (int c = 1; c < GC; ++c) mxa = fmaxf(mxa, mx[c]);
      }
      const float m_new = fmaxf(m, mxa * sl2);
      const bool resc = m_new > m + kRescaleLog2;
      const float alpha = resc ? ex2(m - m_new) : 1.f;
      if (resc) {
        l *= alpha;
        m = m_new;
      }
      const bool rescale_o = cnt > 0 && __any_sync(0xffffffffu, resc);
      const float mu = (m == -INFINITY) ? 0.f : m;
      const uint64_t sl2x2 = f2_pack(sl2, sl2), nmux2 = f2_pack(-mu, -mu);
      float ls0 = 0.f, ls1 = 0.f, ls2 = 0.f, ls3 = 0.f;  // row-sum partials
      PhiloxOut rw;
      // P (bf16, two per 32-bit column) overwrites the first BC / 2 columns
      // of this tile's S, whose scores are already in registers (group g's
      // P lands on columns of group 0, which the first pass has read)
#pragma unroll
      for (int g = 0; g < NG; ++g) {
      if (NG > 1) load_group(g);
#pragma unroll
      for (int q = 0; q < GC; ++q) {  // 32 keys -> 16 columns per store
        // packed words overwrite the scores already consumed: group c4 reads
        // sr[q][8 c4 .. 8 c4 + 7] and writes sr[q][4 c4 .. 4 c4 + 3]
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          float e[8];
#pragma unroll
          for (int j = 0; j < 8; j += 2) {  // exponent arguments of two keys per FMA
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[q][8 * c4 + j]),
                                     __uint_as_float(sr[q][8 * c4 + j + 1])),
                             sl2x2, nmux2),
                      e[j], e[j + 1]);
            e[j] = ex2(e[j]);
            e[j + 1] = ex2(e[j + 1]);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) sr[q][4 * c4 + j] = pack_bf16(e[2 * j], e[2 * j + 1]);
          // l sums the same bf16-rounded weights the PV MMA consumes, so a
          // dominant key's rounding cancels in O / l
          acc_bf16x2(ls0, ls1, sr[q][4 * c4]);
          acc_bf16x2(ls2, ls3, sr[q][4 * c4 + 1]);
          acc_bf16x2(ls0, ls1, sr[q][4 * c4 + 2]);
          acc_bf16x2(ls2, ls3, sr[q][4 * c4 + 3]);
          if (DROP) {
            // dropped weights leave the PV product (l keeps them); one
            // generator call covers keys 32 q + 16 (c4 / 2) .. + 15
            if ((c4 & 1) == 0) rw = rng.group((kbase + g * GW) / 16 + 2 * q + (c4 >> 1), qrow, bh);
            const uint32_t m0 = DropoutRng::keep_bytes(rw.w[2 * (c4 & 1)], rng.t4);
            const uint32_t m1 = DropoutRng::keep_bytes(rw.w[2 * (c4 & 1) + 1], rng.t4);
            sr[q][4 * c4] &= pair_mask(m0, 0);
            sr[q][4 * c4 + 1] &= pair_mask(m0, 1);
            sr[q][4 * c4 + 2] &= pair_mask(m1, 0);
            sr[q][4 * c4 + 3] &= pair_mask(m1, 1);
          }
        }
        tmem_st16(tP + g * (GW / 2) + 16 * q, *reinterpret_cast<const uint32_t(*)[16]>(&sr[q][0]));
      }
      }
      // rescale O only after P is out of the registers (lower register pressure)
      if (rescale_o) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_ld_wait();
          reg_fence(o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          tmem_st32(tO + 32 * c, o);
        }
        tmem_st_wait();
      }
      tmem_st_wait();
      l += (ls0 + ls1) + (ls2 + ls3);
      tc_fence_before();
      mbar_arrive(bar(L::B_PF + s));
      ++cnt;
    }
    // ---------------------------------------------------- epilogue
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_OF), 0, wc));
    tc_fence_after();
    if (ok && active) {
      const int qrow0 = qt * kTile + q4 * 32;  // this warp's first query row
      const int nrows = min(32, N - qrow0);
      uint8_t* obase = static_cast<uint8_t*>(p.o) +
                       (static_cast<size_t>(zq) * slice_rows + row0 + qrow0) *
                           static_cast<size_t>(D) * 2;
      const bool store = qrow < N;
      const bool has = cnt > 0 && l > 0.f;
      // inverted dropout scales the kept weights by 1 / (1 - p')
      const float inv = has ? (DROP ? p.drop.scale : 1.f) / l : 0.f;
      // Each thread packs 64 columns of its O row (128 bytes) into this
      // warp's rows of Q_s (free: the tile's last S product has completed),
      // then each store writes 4 whole 128-byte row pieces.
      const uint32_t stg = sb + L::Q + s * L::TILE + q4 * 4096;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t o[2][32];
        if (cnt > 0) {
          tmem_ld32(tO + 64 * c, o[0]);
          tmem_ld32(tO + 64 * c + 32, o[1]);
          tmem_ld_wait();
          reg_fence(o[0]);
          reg_fence(o[1]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[0][j] = o[1][j] = 0u;
        }
        const uint32_t st = stg + c * L::CHUNK;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint32_t* x = &o[v >> 2][8 * (v & 3)];
          st_shared_v4(st + sw128_offset(lane, v),
                       pack_bf16(__uint_as_float(x[0]) * inv, __uint_as_float(x[1]) * inv),
                       pack_bf16(__uint_as_float(x[2]) * inv, __uint_as_float(x[3]) * inv),
                       pack_bf16(__uint_as_float(x[4]) * inv, __uint_as_float(x[5]) * inv),
                       pack_bf16(__uint_as_float(x[6]) * inv, __uint_as_float(x[7]) * inv));
        }
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int j = 4 * it + (lane >> 3), cc = lane & 7;
          const uint4 v = ld_shared_v4(st + sw128_offset(j, cc));
          if (j < nrows)
            *reinterpret_cast<uint4*>(obase + static_cast<size_t>(j) * D * 2 + c * 128 + cc * 16) = v;
        }
      }
      if (store)
        p.lse[static_cast<size_t>(zq) * slice_rows + row0 + qrow] =
            has ? (m + lg2(l)) * kLn2 : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TCOLS);
  }
}

template <int D, int KIND, int NS_ = 0, int BC = kTile, bool CMP = false>
cudaError_t launch_fwd_d(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, cudaStream_t stream) {
  using L = FwdSmem<D, NS_, BC, CMP>;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = smem_attr_once(
      attr_done, reinterpret_cast<const void*>(fa_fwd_kernel<D, KIND, NS_, BC, CMP>), L::ALLOC);
  if (e != cudaSuccess) return e;
  const int nT = (p.N + kTile - 1) / kTile;
  const int npairs = L::NQT == 1 ? nT : (nT + 1) / 2;
  const long long ctas = static_cast<long long>(npairs) * p.B * p.H;
  return launch_pdl(fa_fwd_kernel<D, KIND, NS_, BC, CMP>, dim3(static_cast<unsigned>(ctas)),
                    dim3(L::THREADS), L::ALLOC, stream, tq, tk, tv, p);
}

}  // namespace

// Block-size sweep configurations: (head dim, key tile, K/V ring stages).
// Shared memory: two query tiles (2 x 128 x d x 2 B) plus `stages` ring
// slots of one key or value tile each (key tile x d x 2 B).  TMEM: S (key
// tile columns) and O (d columns) per query tile, at most 512 columns, so a
// 256-key tile holds one query tile per CTA.
cudaError_t launch_forward_config(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, int kv_stages, int key_tile,
                                  cudaStream_t stream) {
  const int code = p.d * 100000 + key_tile * 100 + kv_stages;
  if (p.single_tile) {  // one query tile per CTA: the compact form
    switch (code) {
      case 12812802: return launch_fwd_d<128, kPlain, 2, 128, true>(p, tq, tk, tv, stream);
      case 12812803: return launch_fwd_d<128, kPlain, 3, 128, true>(p, tq, tk, tv, stream);
      case 12812804: return launch_fwd_d<128, kPlain, 4, 128, true>(p, tq, tk, tv, stream);
      case 12812805: return launch_fwd_d<128, kPlain, 5, 128, true>(p, tq, tk, tv, stream);
      case 12806404: return launch_fwd_d<128, kPlain, 4, 64, true>(p, tq, tk, tv, stream);
      case 12806408: return launch_fwd_d<128, kPlain, 8, 64, true>(p, tq, tk, tv, stream);
      case 12825602: return launch_fwd_d<128, kPlain, 2, 256, true>(p, tq, tk, tv, stream);
      case 6412802: return launch_fwd_d<64, kPlain, 2, 128, true>(p, tq, tk, tv, stream);
      case 6412804: return launch_fwd_d<64, kPlain, 4, 128, true>(p, tq, tk, tv, stream);
      case 6412808: return launch_fwd_d<64, kPlain, 8, 128, true>(p, tq, tk, tv, stream);
      case 6406408: return launch_fwd_d<64, kPlain, 8, 64, true>(p, tq, tk, tv, stream);
      case 6406416: return launch_fwd_d<64, kPlain, 16, 64, true>(p, tq, tk, tv, stream);
      case 6425602: return launch_fwd_d<64, kPlain, 2, 256, true>(p, tq, tk, tv, stream);
      case 6425604: return launch_fwd_d<64, kPlain, 4, 256, true>(p, tq, tk, tv, stream);
    }
    return cudaErrorInvalidValue;
  }
  switch (code) {
    case 12812802: return launch_fwd_d<128, kPlain, 2>(p, tq, tk, tv, stream);
    case 12812803: return launch_fwd_d<128, kPlain, 3>(p, tq, tk, tv, stream);
    case 12812804: return launch_fwd_d<128, kPlain, 4>(p, tq, tk, tv, stream);
    case 12812805: return launch_fwd_d<128, kPlain, 5>(p, tq, tk, tv, stream);
    case 12806404: return launch_fwd_d<128, kPlain, 4, 64>(p, tq, tk, tv, stream);
    case 12806408: return launch_fwd_d<128, kPlain, 8, 64>(p, tq, tk, tv, stream);
    case 6412802: return launch_fwd_d<64, kPlain, 2>(p, tq, tk, tv, stream);
    case 6412804: return launch_fwd_d<64, kPlain, 4>(p, tq, tk, tv, stream);
    case 6412808: return launch_fwd_d<64, kPlain, 8>(p, tq, tk, tv, stream);
    case 6406408: return launch_fwd_d<64, kPlain, 8, 64>(p, tq, tk, tv, stream);
    case 6406416: return launch_fwd_d<64, kPlain, 16, 64>(p, tq, tk, tv, stream);
  }
  return cudaErrorInvalidValue;
}

template <int D, bool CMP>
cudaError_t launch_forward_kind(int kind, const FwdParams& p, const CUtensorMap& tq,
                                const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t stream) {
  if (kind == kGeneralDropout)
    return launch_fwd_d<D, kGeneralDropout, 0, kTile, CMP>(p, tq, tk, tv, stream);
  if (kind == kGeneral) return launch_fwd_d<D, kGeneral, 0, kTile, CMP>(p, tq, tk, tv, stream);
  if (kind == kGrouped) return launch_fwd_d<D, kGrouped, 0, kTile, CMP>(p, tq, tk, tv, stream);
  return launch_fwd_d<D, kPlain, 0, kTile, CMP>(p, tq, tk, tv, stream);
}

cudaError_t launch_forward(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t stream) {
  const int kind = p.drop.t ? kGeneralDropout
                   : p.cu_seqlens ? kGeneral
                   : (p.Hkv > 0 && p.Hkv != p.H) ? kGrouped : kPlain;
  // Small grids (at most four waves of two-tile CTAs: BERT- or GPT-2-sized
  // batches) run the compact form, one query tile per CTA and two CTAs per
  // SM: one CTA's start and end overlap the other's steps, and the finer
  // grain evens out the last wave (measured: B8 H12 N1024 causal d = 64
  // forward 33.2 -> 29.6 us, B8 H16 N512 20.2 -> 19.4 us; at B4 H16 N4096 the
  // two-tile form is 4 % faster at d = 64 and 8 % at d = 128).
  // Block masks also run the compact form at every size: a two-tile CTA
  // walks the union of its two query tiles' kept key tiles, and with
  // scattered masks most of those steps hold one tile only (one MMA chain
  // per SM instead of two).
  const int nT = (p.N + kTile - 1) / kTile;
  const long long pairs = static_cast<long long>((nT + 1) / 2) * p.B * p.H;
  const int sms = sm_count();
  const bool compact = p.lists.row_ptr != nullptr || (sms > 0 && pairs <= 4LL * sms);
  if (p.d == 64)
    return compact ? launch_forward_kind<64, true>(kind, p, tq, tk, tv, stream)
                   : launch_forward_kind<64, false>(kind, p, tq, tk, tv, stream);
  if (p.d == 128)
    return compact ? launch_forward_kind<128, true>(kind, p, tq, tk, tv, stream)
                   : launch_forward_kind<128, false>(kind, p, tq, tk, tv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
