// Small kernels around the two attention kernels: the block-mask -> tile
// list builder, the backward preprocess (D = rowsum(dO o O), zero dQ
// accumulator) and dQ conversion, the schedule export used by the tests,
// a one-tile tcgen05 probe, and the bounded-wait probe.
#include <math.h>
#include <stdint.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_sched.cuh"

namespace fa {

// ------------------------------------------------------------------ lists
// CSR: for each query tile the ascending key tiles whose mask byte is
// nonzero; CSC: for each key tile the ascending query tiles ("Block-sparse
// FlashAttention": only nonzero blocks are visited).  One CTA of 32 warps
// per mask head reads the mask in chunks of 16 columns (one 16-byte load
// when the mask is 16-byte aligned and nT is a multiple of 16, else byte
// loads), so that a warp covers 512 consecutive columns per access:
//   CSR  a warp per row: row counts, then each lane places its chunk's
//        columns after a prefix over the warp's lanes;
//   CSC  warps split into 512-column strips x row ranges: per-range column
//        counts, a prefix over ranges per column, then each lane walks its
//        16 columns down its row range in ascending order.
// Counts and prefix sums live in shared memory: 2 (nT + 1) + R nT ints, R
// row ranges per strip (R nT <= 32 * 512 + 31 nT).
constexpr int kListWarps = 32;

struct ListLayout {
  int nT, strips, ranges, rows_per_range;
  __host__ __device__ static ListLayout of(int nT) {
    ListLayout L;
    L.nT = nT;
    L.strips = (nT + 511) / 512;
    L.ranges = kListWarps / L.strips > 0 ? kListWarps / L.strips : 1;
    L.rows_per_range = (nT + L.ranges - 1) / L.ranges;
    return L;
  }
  __host__ __device__ int smem_ints() const { return 2 * (nT + 1) + ranges * nT; }
};

// nonzero bits of columns c0 .. c0 + 15 of a mask row (bit k: column c0 + k;
// columns >= nT read as zero)
FA_DEV uint32_t chunk_bits(const uint8_t* row, int c0, int nT, bool vec) {
  if (vec && c0 + 16 <= nT) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + c0));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t bits = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // 0xFF in each nonzero byte, then byte k -> bit k (one multiply moves
      // the four low bits of the bytes to bits 28..31 with no carries)
      const uint32_t nz = __vcmpne4(w[i], 0u);
      bits |= (((nz & 0x01010101u) * 0x10204080u) >> 28) << (4 * i);
    }
    return bits;
  }
  uint32_t bits = 0;
  for (int k = 0; k < 16 && c0 + k < nT; ++k) bits |= (row[c0 + k] != 0 ? 1u : 0u) << k;
  return bits;
}

// exclusive prefix sum of a[0 .. n) in place, a[n] = total (whole block)
FA_DEV void block_exclusive_scan(int* a, int n, int* warp_tot) {
  const int t = threadIdx.x, nthr = blockDim.x, lane = t & 31, warp = t >> 5;
  const int per = (n + nthr - 1) / nthr;
  const int b = t * per, e = min(n, b + per);
  int local = 0;
  for (int i = b; i < e; ++i) local += a[i];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (nthr >> 5) ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += x;
    }
    if (lane < (nthr >> 5)) warp_tot[lane] = wi - w;  // exclusive warp offsets
    if (lane == 31) warp_tot[32] = wi;                 // block total
  }
  __syncthreads();
  int run = warp_tot[warp] + incl - local;
  for (int i = b; i < e; ++i) {
    const int x = a[i];
    a[i] = run;
    run += x;
  }
  if (t == 0) a[n] = warp_tot[32];
  __syncthreads();
}

__global__ void __launch_bounds__(kListWarps * 32) fa_lists_kernel(
    const uint8_t* __restrict__ mask, int nT, int* row_ptr, int* col_idx, int* col_ptr,
    int* row_idx, int* unit_order, int* nlong) {
  grid_dep_wait();  // the previous kernel's writes are visible from here on
  grid_dep_launch();
  extern __shared__ __align__(16) int lsm[];
  __shared__ int warp_tot[33];
  const ListLayout L = ListLayout::of(nT);
  int* rc = lsm;                 // [nT + 1] row counts -> CSR offsets
  int* cc = rc + (nT + 1);       // [nT + 1] column counts -> CSC offsets
  int* rg = cc + (nT + 1);       // [ranges][nT] per-range column counts -> starts
  const int h = blockIdx.x;
  const uint8_t* m = mask + static_cast<size_t>(h) * nT * nT;
  int* rp = row_ptr + static_cast<size_t>(h) * (nT + 1);
  int* cp = col_ptr + static_cast<size_t>(h) * (nT + 1);
  int* ci = col_idx + static_cast<size_t>(h) * nT * nT;
  int* ri = row_idx + static_cast<size_t>(h) * nT * nT;
  int* uo = unit_order + static_cast<size_t>(h) * nT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool vec = (reinterpret_cast<uintptr_t>(mask) % 16 == 0) && (nT % 16 == 0);
  auto row_of = [&](int r) { return m + static_cast<size_t>(r) * nT; };
  // this warp's CSC strip and row range (warps past strips x ranges idle)
  const int strip = warp % L.strips, range = warp / L.strips;
  const bool csc_warp = range < L.ranges;
  const int col0 = strip * 512 + 16 * lane;
  const int r_lo = csc_warp ? min(nT, range * L.rows_per_range) : 0;
  const int r_hi = csc_warp ? min(nT, r_lo + L.rows_per_range) : 0;

  // ---- counts (the row loops are unrolled so that several rows' loads are
  // in flight at once: one CTA has few warps to hide load latency with)
#pragma unroll 4
  for (int r = warp; r < nT; r += kListWarps) {
    int c = 0;
    for (int c0 = 16 * lane; c0 < nT; c0 += 512) c += __popc(chunk_bits(row_of(r), c0, nT, vec));
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) rc[r] = c;
  }
  {
    int cnt[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) cnt[k] = 0;
    if (csc_warp && col0 < nT) {
      for (int r = r_lo; r < r_hi; ++r) {
        const uint32_t bits = chunk_bits(row_of(r), col0, nT, vec);
#pragma unroll
        for (int k = 0; k < 16; ++k) cnt[k] += (bits >> k) & 1u;
      }
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (col0 + k < nT) rg[range * nT + col0 + k] = cnt[k];
    }
  }
  __syncthreads();
  // per column: starts of each row range, column totals
  for (int c = threadIdx.x; c < nT; c += blockDim.x) {
    int run = 0;
    for (int g = 0; g < L.ranges; ++g) {
      int* x = &rg[g * nT + c];
      const int v = (g * L.rows_per_range < nT) ? *x : 0;
      *x = run;
      run += v;
    }
    cc[c] = run;
  }
  __syncthreads();
  block_exclusive_scan(rc, nT, warp_tot);
  block_exclusive_scan(cc, nT, warp_tot);
  for (int a = threadIdx.x; a <= nT; a += blockDim.x) {
    rp[a] = rc[a];
    cp[a] = cc[a];
  }

  // ---- indices
#pragma unroll 2
  for (int r = warp; r < nT; r += kListWarps) {
    int base = rc[r];
    for (int c0s = 0; c0s < nT; c0s += 512) {
      const int c0 = c0s + 16 * lane;
      const uint32_t bits = c0 < nT ? chunk_bits(row_of(r), c0, nT, vec) : 0u;
      const int n = __popc(bits);
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      int pos = base + incl - n;
      for (uint32_t b = bits; b; b &= b - 1) ci[pos++] = c0 + __ffs(b) - 1;
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (csc_warp && col0 < nT) {
    int pos[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) pos[k] = col0 + k < nT ? cc[col0 + k] + rg[range * nT + col0 + k] : 0;
    for (int r = r_lo; r < r_hi; ++r) {
      const uint32_t bits = chunk_bits(row_of(r), col0, nT, vec);
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if ((bits >> k) & 1u) ri[pos[k]++] = r;
    }
  }
  // ---- backward unit order: key tiles by descending CSC length, ties by
  // index (a key tile's rank counts the tiles that come before it), and how
  // many of them are long (more than twice the mean length: e.g. a kept
  // column of every query tile), which the backward starts first
  __syncthreads();  // the CSC pass has read its starts from rg
  int* cnt = rg + ((4 - ((2 * (nT + 1)) & 3)) & 3);  // 16-byte aligned, [nT4]
  const int nT4 = (nT + 3) & ~3;
  for (int t = threadIdx.x; t < nT4; t += blockDim.x) cnt[t] = t < nT ? cc[t + 1] - cc[t] : -1;
  __shared__ int nlong_s;
  if (threadIdx.x == 0) nlong_s = 0;
  __syncthreads();
  const long long total = cc[nT];
  const int4* c4 = reinterpret_cast<const int4*>(cnt);
  for (int t = threadIdx.x; t < nT; t += blockDim.x) {
    const int ct = cnt[t];
    int rank = 0;
    for (int j4 = 0; j4 < nT4 / 4; ++j4) {
      const int4 v = c4[j4];
      const int j = 4 * j4;
      rank += (v.x > ct) || (v.x == ct && j < t);
      rank += (v.y > ct) || (v.y == ct && j + 1 < t);
      rank += (v.z > ct) || (v.z == ct && j + 2 < t);
      rank += (v.w > ct) || (v.w == ct && j + 3 < t);
    }
    uo[rank] = t;
    if (static_cast<long long>(ct) * nT > 2 * total) atomicAdd(&nlong_s, 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) nlong[h] = nlong_s;
}

cudaError_t launch_build_lists(const uint8_t* mask, int mask_heads, int nT, int* row_ptr,
                               int* col_idx, int* col_ptr, int* row_idx, int* unit_order,
                               int* nlong, cudaStream_t stream) {
  const int smem = ListLayout::of(nT).smem_ints() * static_cast<int>(sizeof(int));
  if (smem > 48 * 1024) {
    static std::atomic<unsigned long long> attr_done{0};
    // the largest layout (nT = 8192) once per device, so that no later call
    // needs to raise it again
    cudaError_t e = smem_attr_once(attr_done, reinterpret_cast<const void*>(fa_lists_kernel),
                                   ListLayout::of(8192).smem_ints() * static_cast<int>(sizeof(int)));
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(fa_lists_kernel, dim3(mask_heads), dim3(kListWarps * 32), smem, stream, mask,
                    nT, row_ptr, col_idx, col_ptr, row_idx, unit_order, nlong);
}

// ------------------------------------------------------------------ backward helpers
// dQ_acc = 0 and D_i = sum_c dO_ic O_ic in fp32.  For D each thread takes
// items of 8 consecutive elements of a row (16-byte loads of O and dO); the
// D/8 threads of a row reduce with shuffles.  Every thread keeps
// kUnroll grid-stride items in flight, and the grid is sized so that each
// thread has about that many.
constexpr int kUnroll = 4;

template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const uint4* __restrict__ o,
                                                         const uint4* __restrict__ dO,
                                                         float* __restrict__ delta,
                                                         float4* __restrict__ dq_acc,
                                                         int* __restrict__ zero_i, long long nzero,
                                                         long long rows) {
  grid_dep_launch();
  constexpr int TPR = D / 8;  // threads per row: 8 or 16
  const long long total = rows * TPR;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  // dQ_acc = 0 first: no kernel before this one can still be using the
  // accumulator (the kernels that read or add into it signal their
  // dependents only on completion), so this runs while the forward finishes
  if (dq_acc) {  // null when dQ does not go through the accumulator
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
         t < 2 * total; t += stride)
      dq_acc[t] = z;
  }
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < nzero;
       t += stride)
    zero_i[t] = 0;  // counters of the backward's split last round
  grid_dep_wait();  // the previous kernel's writes (O) are visible from here on
  // the loop condition is warp-uniform (the warp's first item), so every
  // lane takes part in the shuffles
  for (long long t0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
       t0 - (threadIdx.x & 31) < total; t0 += kUnroll * stride) {
    uint4 a[kUnroll], b[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long t = t0 + u * stride;
      if (t < total) {
        a[u] = o[t];
        b[u] = dO[t];
      } else {
        a[u] = make_uint4(0u, 0u, 0u, 0u);
        b[u] = a[u];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long t = t0 + u * stride;
      float acc = bf16_lo(a[u].x) * bf16_lo(b[u].x) + bf16_hi(a[u].x) * bf16_hi(b[u].x) +
                  bf16_lo(a[u].y) * bf16_lo(b[u].y) + bf16_hi(a[u].y) * bf16_hi(b[u].y) +
                  bf16_lo(a[u].z) * bf16_lo(b[u].z) + bf16_hi(a[u].z) * bf16_hi(b[u].z) +
                  bf16_lo(a[u].w) * bf16_lo(b[u].w) + bf16_hi(a[u].w) * bf16_hi(b[u].w);
#pragma unroll
      for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (t < total && (t % TPR) == 0) delta[t / TPR] = acc;
    }
  }
}

// enough 256-thread blocks for about kUnroll items per thread, at most
// `per_sm` blocks per SM of a 152-SM GPU
static int stream_blocks(long long items, int per_sm) {
  const long long want = (items + 256LL * kUnroll - 1) / (256LL * kUnroll);
  const long long cap = 152LL * per_sm;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

cudaError_t launch_bwd_preprocess(const void* o, const void* dO, float* delta, float* dq_acc,
                                  int* zero_i, long long nzero, long long rows, int d,
                                  cudaStream_t stream) {
  const int blocks = stream_blocks(rows * (d / 8), 8);
  const uint4* o4 = static_cast<const uint4*>(o);
  const uint4* do4 = static_cast<const uint4*>(dO);
  float4* acc4 = reinterpret_cast<float4*>(dq_acc);
  if (d == 64)
    return launch_pdl(fa_bwd_pre_kernel<64>, dim3(blocks), dim3(256), 0, stream, o4, do4, delta,
                      acc4, zero_i, nzero, rows);
  return launch_pdl(fa_bwd_pre_kernel<128>, dim3(blocks), dim3(256), 0, stream, o4, do4, delta,
                    acc4, zero_i, nzero, rows);
}

// dq = bf16(scale * dq_acc), 8 elements per item, kUnroll items in flight
__global__ void __launch_bounds__(256) fa_dq_convert_kernel(const float4* __restrict__ acc,
                                                            uint4* __restrict__ dq, long long n8,
                                                            float scale) {
  grid_dep_wait();  // the previous kernel's writes are visible from here on
  // no early grid_dep_launch: the next kernel may be a preprocess that zeroes
  // this accumulator before its own wait
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n8;
       i0 += kUnroll * stride) {
    float4 a[kUnroll], b[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = i0 + u * stride;
      if (i < n8) {
        a[u] = acc[2 * i];
        b[u] = acc[2 * i + 1];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = i0 + u * stride;
      if (i < n8) {
        uint4 w;
        w.x = pack_bf16(a[u].x * scale, a[u].y * scale);
        w.y = pack_bf16(a[u].z * scale, a[u].w * scale);
        w.z = pack_bf16(b[u].x * scale, b[u].y * scale);
        w.w = pack_bf16(b[u].z * scale, b[u].w * scale);
        dq[i] = w;
      }
    }
  }
}

cudaError_t launch_dq_convert(const float* dq_acc, void* dq, long long n, float scale,
                              cudaStream_t stream) {
  const long long n8 = n / 8;
  return launch_pdl(fa_dq_convert_kernel, dim3(stream_blocks(n8, 8)), dim3(256), 0, stream,
                    reinterpret_cast<const float4*>(dq_acc), static_cast<uint4*>(dq), n8, scale);
}

// ------------------------------------------------------------------ schedule export
// Runs the kernels' own schedule code and writes, per head layout, the key
// tiles each query tile visits in the forward and the query tiles each key
// tile visits in the backward.  lists are [heads][nT][nT], counts [heads][nT].
__global__ void fa_schedule_kernel(int N, int causal, TileLists L, int heads, int* fc, int* bc,
                                   int* fl, int* bl) {
  const int nT = (N + kTile - 1) / kTile, npairs = (nT + 1) / 2;
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long nf = static_cast<long long>(heads) * npairs;
  const long long nb = static_cast<long long>(heads) * nT;
  if (t < nf) {
    const int head = static_cast<int>(t / npairs), pair = static_cast<int>(t % npairs);
    FwdSchedule s;
    s.init(pair, nT, causal != 0, L, head);
    int c0 = 0, c1 = 0, kt, mem;
    int* l0 = fl + (static_cast<size_t>(head) * nT + s.qt[0]) * nT;
    int* l1 = fl + (static_cast<size_t>(head) * nT + (s.act[1] ? s.qt[1] : s.qt[0])) * nT;
    while (s.next(kt, mem)) {
      if (mem & 1) l0[c0++] = kt;
      if (mem & 2) l1[c1++] = kt;
    }
    fc[static_cast<size_t>(head) * nT + s.qt[0]] = c0;
    if (s.act[1]) fc[static_cast<size_t>(head) * nT + s.qt[1]] = c1;
  } else if (t < nf + nb) {
    const long long u = t - nf;
    const int head = static_cast<int>(u / nT), kt = static_cast<int>(u % nT);
    BwdSchedule s;
    s.init(kt, nT, causal != 0, L, head);
    int c = 0, qt;
    int* lo = bl + (static_cast<size_t>(head) * nT + kt) * nT;
    while (s.next(qt)) lo[c++] = qt;
    bc[static_cast<size_t>(head) * nT + kt] = c;
  }
}

cudaError_t launch_schedule_export(int N, int causal, const TileLists& lists, int heads,
                                   int* fwd_counts, int* bwd_counts, int* fwd_lists,
                                   int* bwd_lists, cudaStream_t stream) {
  const int nT = (N + kTile - 1) / kTile, npairs = (nT + 1) / 2;
  const long long total = static_cast<long long>(heads) * (npairs + nT);
  const int blocks = static_cast<int>((total + 127) / 128);
  fa_schedule_kernel<<<blocks, 128, 0, stream>>>(N, causal, lists, heads, fwd_counts, bwd_counts,
                                                 fwd_lists, bwd_lists);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ tcgen05 probe
// One CTA, one 128-row tile, the operand forms the attention kernels use:
//   mode 0: C[128x128] = A B^T, A and B [128 x 128] K-major through TMA
//           (the S = Q K^T form)
//   mode 1: C[128xn] = A B, A [128 x 128] written by threads in the 128-byte
//           swizzle, B [128 x n] MN-major through TMA (the O += P V form)
//   mode 2: C[128xn] = A^T B, A [128 x 128] and B [128 x n] both MN-major
//           through TMA (the dV += P^T dO and dK += dS^T Q forms)
//   mode 3: C[128xn] = A B, A [128 x 128] written by threads into TMEM (two
//           bf16 per column), B [128 x n] MN-major through TMA (O += P V with
//           P held in tensor memory)
__global__ void __launch_bounds__(128, 1)
    fa_mma_probe_kernel(const __grid_constant__ CUtensorMap ta,
                        const __grid_constant__ CUtensorMap tb, const uint16_t* a_raw, float* c,
                        int mode, int n, int* err, uint64_t wait_ns) {
  constexpr int CHUNK = 16384;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t A = sb, B = sb + 2 * CHUNK, bar_ld = sb + 4 * CHUNK, bar_mma = bar_ld + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 4 * CHUNK + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 4 * CHUNK + 20);
  const int warp = threadIdx.x >> 5, t = threadIdx.x;
  if (t == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, err, wait_ns};
  const int nb_chunks = (mode == 0) ? 2 : n / 64;
  if (t == 0) {
    const int a_chunks = (mode == 1 || mode == 3) ? 0 : 2;
    mbar_arrive_expect_tx(bar_ld, (a_chunks + nb_chunks) * CHUNK);
    for (int cc = 0; cc < a_chunks; ++cc) tma_load_3d(A + cc * CHUNK, &ta, bar_ld, 64 * cc, 0, 0);
    for (int cc = 0; cc < nb_chunks; ++cc) tma_load_3d(B + cc * CHUNK, &tb, bar_ld, 64 * cc, 0, 0);
  }
  if (mode == 1) {
    // thread t writes row t of A (128 bf16) in the 128-byte swizzle
    const uint4* src = reinterpret_cast<const uint4*>(a_raw + t * 128);
    for (int cc = 0; cc < 16; ++cc) {
      const uint4 w = src[cc];
      st_shared_v4(A + (cc >> 3) * CHUNK + sw128_offset(t, cc & 7), w.x, w.y, w.z, w.w);
    }
    fence_async_smem();
  }
  if (mode == 3) {
    // thread t writes row t of A into TMEM lane t, columns 128..191
    const uint4* src = reinterpret_cast<const uint4*>(a_raw + t * 128);
    for (int half = 0; half < 2; ++half) {
      uint32_t w[32];
      for (int cc = 0; cc < 8; ++cc) {
        const uint4 x = src[8 * half + cc];
        w[4 * cc + 0] = x.x;
        w[4 * cc + 1] = x.y;
        w[4 * cc + 2] = x.z;
        w[4 * cc + 3] = x.w;
      }
      tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 128 + 32 * half, w);
    }
    tmem_st_wait();
    tc_fence_before();
  }
  __syncthreads();
  bool ok = true;
  if (t == 0) {
    ok = wait_bar(bar_ld, 0, wc);
    if (ok) {
      tc_fence_after();
      if (mode == 0) {
        const uint32_t id = idesc_bf16(128, 128, false, false);
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * CHUNK + (kk & 3) * 32;
          mma_bf16_ss(tmem, desc_sw128(A + off, 16, 1024), desc_sw128(B + off, 16, 1024), id,
                      kk > 0);
        }
      } else if (mode == 1) {
        const uint32_t id = idesc_bf16(128, n, false, true);
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * CHUNK + (kk & 3) * 32;
          mma_bf16_ss(tmem, desc_sw128(A + aoff, 16, 1024), desc_sw128(B + kk * 2048, CHUNK, 1024),
                      id, kk > 0);
        }
      } else if (mode == 2) {
        const uint32_t id = idesc_bf16(128, n, true, true);
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ss(tmem, desc_sw128(A + kk * 2048, CHUNK, 1024),
                      desc_sw128(B + kk * 2048, CHUNK, 1024), id, kk > 0);
      } else {
        const uint32_t id = idesc_bf16(128, n, false, true);
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(tmem, tmem + 128 + kk * 8, desc_sw128(B + kk * 2048, CHUNK, 1024), id,
                      kk > 0);
      }
    }
    mma_commit(bar_mma);
    drain_bar(bar_mma, 0, wait_ns);
    if (!ok) drain_bar(bar_ld, 0, wait_ns);
  }
  __syncthreads();
  ok = !*abort_flag;
  tc_fence_after();
  const int ncols = (mode == 0) ? 128 : n;
  if (ok) {
    for (int cc = 0; cc < ncols / 32; ++cc) {
      uint32_t r[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 32 * cc, r);
      tmem_ld_wait();
      reg_fence(r);
      for (int j = 0; j < 32; ++j) c[t * ncols + 32 * cc + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

cudaError_t launch_mma_probe(const CUtensorMap& ta, const CUtensorMap& tb, const void* a_raw,
                             float* c, int mode, int n, int* err, uint64_t wait_ns,
                             cudaStream_t stream) {
  const int smem = 4 * 16384 + 64 + 1024;
  cudaError_t e = cudaFuncSetAttribute(fa_mma_probe_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  fa_mma_probe_kernel<<<1, 128, smem, stream>>>(ta, tb, static_cast<const uint16_t*>(a_raw), c,
                                                mode, n, err, wait_ns);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ wait probe
// Waits on an mbarrier that nothing will ever complete.  The bounded wait
// gives up after wait_ns, records the timeout in the status word and the
// kernel returns normally.
__global__ void fa_wait_probe_kernel(int* err, uint64_t wait_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl wc{&abort_flag, err, wait_ns};
    (void)wait_bar(smem_u32(&bar), 0, wc);
  }
  __syncthreads();
}

cudaError_t launch_wait_probe(int* err, uint64_t wait_ns, cudaStream_t stream) {
  fa_wait_probe_kernel<<<1, 32, 0, stream>>>(err, wait_ns);
  return cudaGetLastError();
}

}  // namespace fa

// ------------------------------------------------------------------ status word
// One per device (each device that loads the module gets its own copy).
__device__ int g_fa_status_word = 0;

namespace fa {
int* status_word_address() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fa_status_word) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}
}  // namespace fa
