// Declarations shared by the library's translation units (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>
#include <stdint.h>

#include <atomic>

namespace fa {

// Dynamic shared memory above 48 KB has to be allowed per kernel, in each
// device's context.  `done` is the kernel's own record, one bit per device
// already set up; a device index of 64 or more is set up on every launch.
inline cudaError_t smem_attr_once(std::atomic<unsigned long long>& done, const void* kernel,
                                  int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// SM count of the current device, read once per device (0 on error).
inline int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cached[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

// Launch with programmatic stream serialization (the kernel starts with
// grid_dep_wait, see fa_ptx.cuh), so that its scheduling overlaps the tail of
// the previous kernel in the stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kTile = 128;  // query rows and keys per tile (Br = Bc = 128)

// Block-sparse tile lists for one mask head layout:
//   csr: row_ptr [mask_heads][nT+1] (head-local offsets),
//        col_idx [mask_heads][nT*nT] (ascending key tiles of each query tile)
//   csc: col_ptr / row_idx, the same for each key tile (ascending query tiles)
//   unit_order [mask_heads][nT]: key tiles by descending CSC length (ties by
//        index): the order in which the backward takes its units
//   nlong [mask_heads]: how many of them are longer than twice the mean
struct TileLists {
  const int* row_ptr = nullptr;
  const int* col_idx = nullptr;
  const int* col_ptr = nullptr;
  const int* row_idx = nullptr;
  const int* unit_order = nullptr;
  const int* nlong = nullptr;
  int mask_heads = 0;
  int nT = 0;
};

// Dropout on P: element (i, j) of (batch, head) slice b*H + h is kept iff
// byte j mod 16 of Philox4x32-10((j/16, i, b*H + h, offset), seed) >= t;
// kept weights are scaled by 256 / (256 - t).  t = 0 means no dropout.
struct DropoutParams {
  uint32_t seed_lo = 0, seed_hi = 0, offset = 0;
  uint32_t t = 0;
  float scale = 1.f;
  // Philox key of round r: (seed_lo + r * 0x9E3779B9, seed_hi + r * 0xBB67AE85),
  // formed on the host; kernel parameters, read by the rounds as constants
  uint32_t rk[20] = {};
};

struct FwdParams {
  void* o = nullptr;      // bf16 [BH, N, d]
  float* lse = nullptr;   // fp32 [BH, N]
  int B = 0, H = 0, N = 0, d = 0;
  int Hkv = 0;            // key/value heads (H % Hkv == 0); 0 means H
  float scale = 0.f;
  int causal = 0;
  TileLists lists;        // sparse when lists.row_ptr != nullptr
  int single_tile = 0;    // 1: one 128-row query tile per CTA instead of two
  // variable-length batch: tensors [H, total, d], sequence b in rows
  // cu_seqlens[b] .. cu_seqlens[b+1] (N is then the longest sequence)
  const int* cu_seqlens = nullptr;
  int total = 0;
  DropoutParams drop;     // dropout on P (kernels of kind kGeneralDropout)
  int* err = nullptr;     // device status word
  uint64_t wait_ns = 0;
};

struct BwdParams {
  const float* lse = nullptr;   // fp32 [BH, N]
  const float* delta = nullptr; // fp32 [BH, N]  D_i = <dO_i, O_i>
  float* dq_acc = nullptr;      // fp32 [BH, N, d] (unscaled sum of dS K)
  void* dk = nullptr;           // bf16 [B*Hkv, N, d]
  void* dv = nullptr;           // bf16 [B*Hkv, N, d]
  int B = 0, H = 0, N = 0, d = 0;
  int Hkv = 0;                  // key/value heads (H % Hkv == 0); 0 means H
  float scale = 0.f;
  int causal = 0;
  TileLists lists;              // sparse when lists.col_ptr != nullptr
  const int* cu_seqlens = nullptr;  // variable-length batch (as FwdParams)
  int total = 0;
  DropoutParams drop;
  int skip_dq = 0;  // 1: no dQ product (dQ comes from the query-tile pass)
  // Split last round: when the last round of units fills at most half the
  // grid, each of its units runs as two halves of its query tiles; the first
  // half to finish parks its fp32 dV, dK ([2][128][d] per slot) in part, the
  // second adds them to its own.  part_cnt: [nslot] arrival counts then
  // [nslot] ready flags, zero on entry.  Null / 0: no split.
  float* part = nullptr;
  int* part_cnt = nullptr;
  int nslot = 0;
  // block mask: next-unit counter (zero on entry; the preprocess zeroes it)
  int* unit_counter = nullptr;
  int* err = nullptr;
  uint64_t wait_ns = 0;
};

// Kernel instantiations: plain, grouped K/V, the general one (variable-length
// or equal-length batch, grouped K/V allowed) and the general one with
// dropout on P.
enum KernelKind : int { kPlain = 0, kGrouped = 1, kGeneral = 2, kGeneralDropout = 3 };

// 3-D bf16 view {d, N, B*H} of a [B, H, N, d] tensor, box_rows x 64-column
// boxes (128 rows except the 64-key tiles of the block-size sweep) with
// 128-byte swizzle.
bool make_tile_map(CUtensorMap* map, const void* base, int BH, int N, int d,
                   int box_rows = kTile);
// 3-D fp32 view {d, N, B*H} of a [B, H, N, d] fp32 tensor, 32 x 32 boxes
// (128-byte rows, 128-byte swizzle): the dQ accumulator for TMA reduce-add.
bool make_acc_map(CUtensorMap* map, const void* base, int BH, int N, int d);

cudaError_t launch_forward(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t stream);
// the forward with a chosen key tile width (64, 128, 256) and K/V ring
// depth; K and V maps must have min(key_tile, 128)-row boxes
cudaError_t launch_forward_config(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, int kv_stages, int key_tile,
                                  cudaStream_t stream);
cudaError_t launch_backward_main(const BwdParams& p, const CUtensorMap& tq,
                                 const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const CUtensorMap& tdq,
                                 cudaStream_t stream);
// Query-tile dQ pass of the deterministic backward (plain layout).
struct DqParams {
  const float* lse = nullptr;
  const float* delta = nullptr;
  void* dq = nullptr;  // bf16 [B, H, N, d], written whole
  int B = 0, H = 0, N = 0, d = 0;
  float scale = 0.f;
  int causal = 0;
  TileLists lists;
  int* err = nullptr;
  uint64_t wait_ns = 0;
};

cudaError_t launch_backward_dq(const DqParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv, const CUtensorMap& tdo,
                               cudaStream_t stream);

cudaError_t launch_bwd_preprocess(const void* o, const void* dO, float* delta, float* dq_acc,
                                  int* zero_i, long long nzero,
                                  long long rows, int d, cudaStream_t stream);
cudaError_t launch_dq_convert(const float* dq_acc, void* dq, long long n, float scale,
                              cudaStream_t stream);
cudaError_t launch_build_lists(const uint8_t* mask, int mask_heads, int nT, int* row_ptr,
                               int* col_idx, int* col_ptr, int* row_idx, int* unit_order,
                               int* nlong, cudaStream_t stream);
// schedule export (tests): per query tile the key tiles the forward visits
// and per key tile the query tiles the backward visits
cudaError_t launch_schedule_export(int N, int causal, const TileLists& lists, int heads,
                                   int* fwd_counts, int* bwd_counts, int* fwd_lists,
                                   int* bwd_lists, cudaStream_t stream);
cudaError_t launch_mma_probe(const CUtensorMap& ta, const CUtensorMap& tb, const void* a_raw,
                             float* c, int mode, int n, int* err, uint64_t wait_ns,
                             cudaStream_t stream);
cudaError_t launch_wait_probe(int* err, uint64_t wait_ns, cudaStream_t stream);

}  // namespace fa
