// Host side of the C ABI: argument checks, TMA descriptors, workspace
// layout, launches and the per-device status word.
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {
int* status_word_address();  // fa_aux.cu
}

namespace {

using fa::kTile;

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
std::atomic<unsigned long long> g_wait_ns{0};

unsigned long long wait_limit_ns() {
  unsigned long long v = g_wait_ns.load();
  if (v == 0) {
    v = kDefaultWaitNs;
    if (const char* e = getenv("FA_WAIT_LIMIT_NS")) {
      const unsigned long long x = strtoull(e, nullptr, 10);
      if (x > 0) v = x;
    }
    g_wait_ns.store(v);
  }
  return v;
}

// status word address per device, looked up once per device
constexpr int kMaxDevices = 64;
std::atomic<int*> g_status[kMaxDevices];
std::mutex g_status_mu;

int* status_word(fa_status* st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *st = FA_ERR_CUDA;
    return nullptr;
  }
  int* p = g_status[dev].load();
  if (p) return p;
  std::lock_guard<std::mutex> lk(g_status_mu);
  p = g_status[dev].load();
  if (!p) {
    p = fa::status_word_address();
    if (!p) {
      *st = FA_ERR_CUDA;
      return nullptr;
    }
    g_status[dev].store(p);
  }
  return p;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

fa_status check_shape(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (!(isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long total = static_cast<long long>(B) * H * N * d;
  if (total >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa_status check_ptr16(const void* p) {
  if (!p) return FA_ERR_INVALID_ARG;
  if (!aligned(p, 16)) return FA_ERR_MISALIGNED;
  return FA_OK;
}

fa_status check_ptr4(const void* p) {
  if (!p) return FA_ERR_INVALID_ARG;
  if (!aligned(p, 4)) return FA_ERR_MISALIGNED;
  return FA_OK;
}

#define FA_TRY(x)                    \
  do {                               \
    const fa_status _s = (x);        \
    if (_s != FA_OK) return _s;      \
  } while (0)

#define FA_CUDA(x)                                \
  do {                                            \
    if ((x) != cudaSuccess) return FA_ERR_CUDA;   \
  } while (0)

int num_tiles(int N) { return (N + kTile - 1) / kTile; }

struct BwdWorkspace {
  float* delta;
  float* dq_acc;
  float* part;     // split-last-round partials: [nslot][2][128][d] fp32
  int* part_cnt;   // [2 * nslot]
  int* unit_counter;  // [1] next unit of the block-sparse backward
  int nslot;
};

// Slots for the split last round (the d = 128 kernel only): the last round
// splits only when it holds at most half the grid, so at most units / 2 (and
// 96, half of 192 SMs).
int split_slots(int B, int H, int N, int d) {
  if (d != 128) return 0;
  const long long units = static_cast<long long>(B) * H * num_tiles(N);
  return units > 64 ? static_cast<int>(units / 2 < 96 ? units / 2 : 96) : 0;
}

size_t bwd_ws_bytes(int B, int H, int N, int d) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t ns = static_cast<size_t>(split_slots(B, H, N, d));
  return align256(rows * sizeof(float)) + align256(rows * d * sizeof(float)) +
         align256(ns * 2 * kTile * d * sizeof(float)) + align256((2 * ns + 1) * sizeof(int));
}

BwdWorkspace bwd_ws(void* ws, int B, int H, int N, int d) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  BwdWorkspace w;
  char* base = static_cast<char*>(ws);
  w.delta = reinterpret_cast<float*>(base);
  base += align256(rows * sizeof(float));
  w.dq_acc = reinterpret_cast<float*>(base);
  base += align256(rows * d * sizeof(float));
  w.nslot = split_slots(B, H, N, d);
  w.part = reinterpret_cast<float*>(base);
  base += align256(static_cast<size_t>(w.nslot) * 2 * kTile * d * sizeof(float));
  w.part_cnt = reinterpret_cast<int*>(base);
  w.unit_counter = w.part_cnt + 2 * w.nslot;
  return w;
}

size_t lists_bytes(int N, int mask_heads) {
  const size_t nT = static_cast<size_t>(num_tiles(N));
  return align256(sizeof(int) * mask_heads * (2 * (nT + 1) + 2 * nT * nT + nT + 1));
}

fa::TileLists lists_in(void* ws, int N, int mask_heads) {
  const size_t nT = static_cast<size_t>(num_tiles(N));
  int* base = static_cast<int*>(ws);
  fa::TileLists L;
  L.row_ptr = base;
  L.col_ptr = base + mask_heads * (nT + 1);
  L.col_idx = base + 2 * mask_heads * (nT + 1);
  L.row_idx = L.col_idx + mask_heads * nT * nT;
  L.unit_order = L.row_idx + mask_heads * nT * nT;
  L.nlong = L.unit_order + mask_heads * nT;
  L.mask_heads = mask_heads;
  L.nT = static_cast<int>(nT);
  return L;
}

fa_status build_lists(const uint8_t* mask, int mask_heads, int N, void* ws, cudaStream_t stream) {
  fa::TileLists L = lists_in(ws, N, mask_heads);
  FA_CUDA(fa::launch_build_lists(mask, mask_heads, L.nT, const_cast<int*>(L.row_ptr),
                                 const_cast<int*>(L.col_idx), const_cast<int*>(L.col_ptr),
                                 const_cast<int*>(L.row_idx), const_cast<int*>(L.unit_order),
                                 const_cast<int*>(L.nlong), stream));
  return FA_OK;
}

fa_status check_mask(const uint8_t* mask, int mask_heads, int H, int N) {
  if (!mask) return FA_ERR_INVALID_ARG;
  if (mask_heads != 1 && mask_heads != H) return FA_ERR_INVALID_ARG;
  if (num_tiles(N) > 8192) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Packed variable-length batch: tensors [H, total, d], sequence b in rows
// cu_seqlens[b] .. cu_seqlens[b+1] (device array), N = the longest length.
struct Varlen {
  const int* cu_seqlens = nullptr;
  int total = 0;
};

fa_status forward_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int Hkv, int N, int d, float scale, int causal,
                       const fa::TileLists* lists, cudaStream_t stream,
                       const Varlen& vl = Varlen(),
                       const fa::DropoutParams& drop = fa::DropoutParams()) {
  fa_status st = FA_OK;
  int* err = status_word(&st);
  if (!err) return st;
  // TMA slices: (batch, head) pairs of N rows, or heads of `total` rows
  const int zq = vl.cu_seqlens ? H : B * H, zkv = vl.cu_seqlens ? Hkv : B * Hkv;
  const int rows = vl.cu_seqlens ? vl.total : N;
  CUtensorMap tq, tk, tv;
  if (!fa::make_tile_map(&tq, q, zq, rows, d) || !fa::make_tile_map(&tk, k, zkv, rows, d) ||
      !fa::make_tile_map(&tv, v, zkv, rows, d))
    return FA_ERR_CUDA;
  fa::FwdParams p;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.N = N;
  p.d = d;
  p.scale = scale;
  p.causal = causal ? 1 : 0;
  if (lists) p.lists = *lists;
  p.cu_seqlens = vl.cu_seqlens;
  p.total = vl.total;
  p.drop = drop;
  p.err = err;
  p.wait_ns = wait_limit_ns();
  FA_CUDA(fa::launch_forward(p, tq, tk, tv, stream));
  return FA_OK;
}

fa_status backward_main_impl(const void* q, const void* k, const void* v, const void* dO,
                             const float* lse, void* dk, void* dv, int B, int H, int Hkv, int N,
                             int d, float scale, int causal, const BwdWorkspace& w,
                             const fa::TileLists* lists, cudaStream_t stream,
                             const Varlen& vl = Varlen(),
                             const fa::DropoutParams& drop = fa::DropoutParams()) {
  fa_status st = FA_OK;
  int* err = status_word(&st);
  if (!err) return st;
  const int zq = vl.cu_seqlens ? H : B * H, zkv = vl.cu_seqlens ? Hkv : B * Hkv;
  const int rows = vl.cu_seqlens ? vl.total : N;
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!fa::make_tile_map(&tq, q, zq, rows, d) || !fa::make_tile_map(&tk, k, zkv, rows, d) ||
      !fa::make_tile_map(&tv, v, zkv, rows, d) || !fa::make_tile_map(&tdo, dO, zq, rows, d) ||
      !fa::make_acc_map(&tdq, w.dq_acc, zq, rows, d))
    return FA_ERR_CUDA;
  fa::BwdParams p;
  p.lse = lse;
  p.delta = w.delta;
  p.dq_acc = w.dq_acc;
  p.dk = dk;
  p.dv = dv;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.N = N;
  p.d = d;
  p.scale = scale;
  p.causal = causal ? 1 : 0;
  if (lists) p.lists = *lists;
  p.cu_seqlens = vl.cu_seqlens;
  p.total = vl.total;
  p.drop = drop;
  p.unit_counter = w.unit_counter;
  if (!lists && w.nslot > 0) {  // the split last round (not with a block mask)
    p.part = w.part;
    p.part_cnt = w.part_cnt;
    p.nslot = w.nslot;
  }
  p.err = err;
  p.wait_ns = wait_limit_ns();
  FA_CUDA(fa::launch_backward_main(p, tq, tk, tv, tdo, tdq, stream));
  return FA_OK;
}

fa_status check_fwd_args(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int d, float scale) {
  FA_TRY(check_shape(B, H, N, d, scale));
  FA_TRY(check_ptr16(q));
  FA_TRY(check_ptr16(k));
  FA_TRY(check_ptr16(v));
  FA_TRY(check_ptr16(o));
  FA_TRY(check_ptr4(lse));
  return FA_OK;
}

fa_status check_bwd_args(const void* q, const void* k, const void* v, const void* o,
                         const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, float scale) {
  FA_TRY(check_shape(B, H, N, d, scale));
  for (const void* p : {q, k, v, o, dO, static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv)})
    FA_TRY(check_ptr16(p));
  FA_TRY(check_ptr4(lse));
  return FA_OK;
}

fa_status check_groups(int H, int Hkv) {
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Packed variable-length batch: B sequences, the longest max_seqlen rows,
// `total` rows in all.  cu_seqlens lives on the device and is not read here;
// the kernels clamp its entries to [0, total], so a malformed array gives
// undefined values but no access outside the tensors.
fa_status check_varlen(const int* cu_seqlens, int B, int max_seqlen, int total, int H, int d,
                       float scale) {
  if (B < 1 || H < 1 || total < 0 || max_seqlen < 0) return FA_ERR_INVALID_ARG;
  if (!(isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  FA_TRY(check_ptr4(cu_seqlens));
  if (total > 0 && (max_seqlen < 1 || max_seqlen > total)) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(H) * total * d >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * num_tiles(max_seqlen) >= (1LL << 31))
    return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Dropout probability p in [0, 1) -> threshold t = rint(256 p) (p taken in
// float32, the product in double) and scale 256 / (256 - t); t = 256 (all
// dropped) is refused.
fa_status make_dropout(float p_drop, unsigned long long seed, unsigned offset,
                       fa::DropoutParams* out) {
  if (!(p_drop >= 0.f && p_drop < 1.f)) return FA_ERR_INVALID_ARG;
  const double t = nearbyint(256.0 * static_cast<double>(p_drop));
  if (t >= 256.0) return FA_ERR_INVALID_ARG;
  out->t = static_cast<uint32_t>(t);
  out->scale = static_cast<float>(256.0 / (256.0 - t));
  out->seed_lo = static_cast<uint32_t>(seed);
  out->seed_hi = static_cast<uint32_t>(seed >> 32);
  out->offset = offset;
  for (uint32_t r = 0; r < 10; ++r) {
    out->rk[2 * r] = out->seed_lo + r * 0x9E3779B9u;
    out->rk[2 * r + 1] = out->seed_hi + r * 0xBB67AE85u;
  }
  return FA_OK;
}

// Configurations of the block-size sweep: (d, key tile) -> K/V ring
// stages; a 256-key tile leaves TMEM room for one 128-row query tile only.
bool sweep_config_ok(int d, int rows_per_cta, int key_tile, int kv_stages) {
  if (rows_per_cta != 128 && rows_per_cta != 256) return false;
  if (key_tile == 256 && rows_per_cta != 128) return false;
  if (d == 128) {
    if (key_tile == 128) return kv_stages >= 2 && kv_stages <= 5;
    if (key_tile == 64) return kv_stages == 4 || kv_stages == 8;
    if (key_tile == 256) return kv_stages == 2;
  } else if (d == 64) {
    if (key_tile == 128) return kv_stages == 2 || kv_stages == 4 || kv_stages == 8;
    if (key_tile == 64) return kv_stages == 8 || kv_stages == 16;
    if (key_tile == 256) return kv_stages == 2 || kv_stages == 4;
  }
  return false;
}

fa_status check_ws(void* ws, size_t have, size_t need) {
  if (!ws) return FA_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return FA_ERR_MISALIGNED;
  if (have < need) return FA_ERR_WORKSPACE;
  return FA_OK;
}

// Encoded tensor maps are a pure function of (base, element type, BH, N,
// d): a small per-thread cache returns the same 128 bytes without calling
// the driver again when a caller repeats its buffers (every training step
// does).  Direct-mapped, 16 entries per thread, no locking.
struct MapKey {
  const void* base;
  int BH, N, d, fp32, box_rows;
  bool operator==(const MapKey& o) const {
    return base == o.base && BH == o.BH && N == o.N && d == o.d && fp32 == o.fp32 &&
           box_rows == o.box_rows;
  }
};
struct MapSlot {
  MapKey key;
  CUtensorMap map;
  bool valid;
};
constexpr int kMapSlots = 16;
thread_local MapSlot t_maps[kMapSlots];

int map_slot(const MapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.base) >> 8;
  h ^= static_cast<uint64_t>(k.BH) * 0x9E3779B97F4A7C15ull;
  h ^= static_cast<uint64_t>(k.N) * 0xC2B2AE3D27D4EB4Full;
  h ^= static_cast<uint64_t>(k.d * 2 + k.fp32 + 1024 * k.box_rows) * 0x165667B19E3779F9ull;
  h ^= h >> 29;
  return static_cast<int>(h % kMapSlots);
}

bool encode_map(CUtensorMap* map, const MapKey& key) {
  MapSlot& slot = t_maps[map_slot(key)];
  if (slot.valid && slot.key == key) {
    *map = slot.map;
    return true;
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t esz = key.fp32 ? 4 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(key.d), static_cast<cuuint64_t>(key.N),
                              static_cast<cuuint64_t>(key.BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(key.d) * esz,
                                 static_cast<cuuint64_t>(key.N) * key.d * esz};
  // bf16: box_rows x 64-column boxes; fp32 accumulator: 32 x 32 boxes (both
  // 128-byte rows, 128-byte swizzle)
  const cuuint32_t box_bf16[3] = {64, static_cast<cuuint32_t>(key.box_rows), 1};
  const cuuint32_t box_f32[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const bool ok =
      fn(map, key.fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
         const_cast<void*>(key.base), dims, strides, key.fp32 ? box_f32 : box_bf16, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  if (ok) {
    slot.key = key;
    slot.map = *map;
    slot.valid = true;
  }
  return ok;
}

}  // namespace

namespace fa {
bool make_tile_map(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows) {
  return encode_map(map, MapKey{base, BH, N, d, 0, box_rows});
}
bool make_acc_map(CUtensorMap* map, const void* base, int BH, int N, int d) {
  return encode_map(map, MapKey{base, BH, N, d, 1, 32});
}
}  // namespace fa

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported size or head dimension";
    case FA_ERR_MISALIGNED: return "misaligned pointer";
    case FA_ERR_WORKSPACE: return "workspace too small";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int N, int d, float scale, int causal, cudaStream_t stream) {
  FA_TRY(check_fwd_args(q, k, v, o, lse, B, H, N, d, scale));
  return forward_impl(q, k, v, o, lse, B, H, H, N, d, scale, causal, nullptr, stream);
}

fa_status fa_forward_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int Hkv, int N, int d, float scale, int causal,
                         cudaStream_t stream) {
  FA_TRY(check_fwd_args(q, k, v, o, lse, B, H, N, d, scale));
  FA_TRY(check_groups(H, Hkv));
  return forward_impl(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, nullptr, stream);
}

size_t fa_backward_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  return bwd_ws_bytes(B, H, N, d);
}

fa_status fa_backward_preprocess(const void* o, const void* dO, int B, int H, int N, int d,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  FA_TRY(check_shape(B, H, N, d, 1.f));
  FA_TRY(check_ptr16(o));
  FA_TRY(check_ptr16(dO));
  FA_TRY(check_ws(workspace, workspace_bytes, bwd_ws_bytes(B, H, N, d)));
  const BwdWorkspace w = bwd_ws(workspace, B, H, N, d);
  FA_CUDA(fa::launch_bwd_preprocess(o, dO, w.delta, w.dq_acc, w.part_cnt, 2LL * w.nslot + 1,
                                    static_cast<long long>(B) * H * N, d, stream));
  return FA_OK;
}

fa_status fa_backward_main(const void* q, const void* k, const void* v, const void* dO,
                           const float* lse, void* dk, void* dv, int B, int H, int N, int d,
                           float scale, int causal, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  FA_TRY(check_shape(B, H, N, d, scale));
  for (const void* p : {q, k, v, dO, static_cast<const void*>(dk), static_cast<const void*>(dv)})
    FA_TRY(check_ptr16(p));
  FA_TRY(check_ptr4(lse));
  FA_TRY(check_ws(workspace, workspace_bytes, bwd_ws_bytes(B, H, N, d)));
  return backward_main_impl(q, k, v, dO, lse, dk, dv, B, H, H, N, d, scale, causal,
                            bwd_ws(workspace, B, H, N, d), nullptr, stream);
}

fa_status fa_backward_dq_convert(void* dq, int B, int H, int N, int d, float scale,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  FA_TRY(check_shape(B, H, N, d, scale));
  FA_TRY(check_ptr16(dq));
  FA_TRY(check_ws(workspace, workspace_bytes, bwd_ws_bytes(B, H, N, d)));
  const BwdWorkspace w = bwd_ws(workspace, B, H, N, d);
  FA_CUDA(fa::launch_dq_convert(w.dq_acc, dq, static_cast<long long>(B) * H * N * d, scale, stream));
  return FA_OK;
}

fa_status fa_backward(const void* q, const void* k, const void* v, const void* o, const void* dO,
                      const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                      float scale, int causal, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  FA_TRY(check_bwd_args(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale));
  FA_TRY(check_ws(workspace, workspace_bytes, bwd_ws_bytes(B, H, N, d)));
  FA_TRY(fa_backward_preprocess(o, dO, B, H, N, d, workspace, workspace_bytes, stream));
  FA_TRY(fa_backward_main(q, k, v, dO, lse, dk, dv, B, H, N, d, scale, causal, workspace,
                          workspace_bytes, stream));
  return fa_backward_dq_convert(dq, B, H, N, d, scale, workspace, workspace_bytes, stream);
}

fa_status fa_backward_gqa(const void* q, const void* k, const void* v, const void* o,
                          const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                          int H, int Hkv, int N, int d, float scale, int causal, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  FA_TRY(check_bwd_args(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale));
  FA_TRY(check_groups(H, Hkv));
  FA_TRY(check_ws(workspace, workspace_bytes, bwd_ws_bytes(B, H, N, d)));
  FA_TRY(fa_backward_preprocess(o, dO, B, H, N, d, workspace, workspace_bytes, stream));
  FA_TRY(backward_main_impl(q, k, v, dO, lse, dk, dv, B, H, Hkv, N, d, scale, causal,
                            bwd_ws(workspace, B, H, N, d), nullptr, stream));
  return fa_backward_dq_convert(dq, B, H, N, d, scale, workspace, workspace_bytes, stream);
}

fa_status fa_forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens, int B, int max_seqlen, int total, int H,
                            int Hkv, int d, float scale, int causal, float p_drop,
                            unsigned long long seed, unsigned offset, cudaStream_t stream) {
  FA_TRY(check_varlen(cu_seqlens, B, max_seqlen, total, H, d, scale));
  FA_TRY(check_groups(H, Hkv));
  fa::DropoutParams drop;
  FA_TRY(make_dropout(p_drop, seed, offset, &drop));
  for (const void* p : {q, k, v, static_cast<const void*>(o)}) FA_TRY(check_ptr16(p));
  FA_TRY(check_ptr4(lse));
  if (total == 0) return FA_OK;  // every sequence empty: nothing to write
  Varlen vl;
  vl.cu_seqlens = cu_seqlens;
  vl.total = total;
  return forward_impl(q, k, v, o, lse, B, H, Hkv, max_seqlen, d, scale, causal, nullptr, stream,
                      vl, drop);
}

fa_status fa_backward_varlen(const void* q, const void* k, const void* v, const void* o,
                             const void* dO, const float* lse, void* dq, void* dk, void* dv,
                             const int* cu_seqlens, int B, int max_seqlen, int total, int H,
                             int Hkv, int d, float scale, int causal, float p_drop,
                             unsigned long long seed, unsigned offset, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  FA_TRY(check_varlen(cu_seqlens, B, max_seqlen, total, H, d, scale));
  FA_TRY(check_groups(H, Hkv));
  fa::DropoutParams drop;
  FA_TRY(make_dropout(p_drop, seed, offset, &drop));
  for (const void* p : {q, k, v, o, dO, static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv)})
    FA_TRY(check_ptr16(p));
  FA_TRY(check_ptr4(lse));
  if (total == 0) return FA_OK;
  // the whole packed batch is one (1, H, total) problem for the row-wise
  // preprocess and the dQ conversion
  FA_TRY(check_ws(workspace, workspace_bytes, bwd_ws_bytes(1, H, total, d)));
  FA_TRY(fa_backward_preprocess(o, dO, 1, H, total, d, workspace, workspace_bytes, stream));
  Varlen vl;
  vl.cu_seqlens = cu_seqlens;
  vl.total = total;
  FA_TRY(backward_main_impl(q, k, v, dO, lse, dk, dv, B, H, Hkv, max_seqlen, d, scale, causal,
                            bwd_ws(workspace, 1, H, total, d), nullptr, stream, vl, drop));
  return fa_backward_dq_convert(dq, 1, H, total, d, scale, workspace, workspace_bytes, stream);
}

fa_status fa_backward_deterministic(const void* q, const void* k, const void* v, const void* o,
                                    const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                    int B, int H, int N, int d, float scale, int causal,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  FA_TRY(check_bwd_args(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale));
  const size_t rows = static_cast<size_t>(B) * H * N;
  FA_TRY(check_ws(workspace, workspace_bytes, align256(rows * sizeof(float))));
  fa_status st = FA_OK;
  int* err = status_word(&st);
  if (!err) return st;
  float* delta = static_cast<float*>(workspace);
  // D only: the dQ accumulator is not used
  FA_CUDA(fa::launch_bwd_preprocess(o, dO, delta, nullptr, nullptr, 0, static_cast<long long>(rows), d,
                                    stream));
  CUtensorMap tq, tk, tv, tdo, tdq;
  // tdq is never dereferenced by the key-tile pass without its dQ product;
  // it only has to be a well-formed map
  if (!fa::make_tile_map(&tq, q, B * H, N, d) || !fa::make_tile_map(&tk, k, B * H, N, d) ||
      !fa::make_tile_map(&tv, v, B * H, N, d) || !fa::make_tile_map(&tdo, dO, B * H, N, d) ||
      !fa::make_acc_map(&tdq, workspace, 1, 32, 32))
    return FA_ERR_CUDA;
  fa::BwdParams p;
  p.lse = lse;
  p.delta = delta;
  p.dk = dk;
  p.dv = dv;
  p.B = B;
  p.H = H;
  p.Hkv = H;
  p.N = N;
  p.d = d;
  p.scale = scale;
  p.causal = causal ? 1 : 0;
  p.skip_dq = 1;
  p.err = err;
  p.wait_ns = wait_limit_ns();
  FA_CUDA(fa::launch_backward_main(p, tq, tk, tv, tdo, tdq, stream));
  fa::DqParams pq;
  pq.lse = lse;
  pq.delta = delta;
  pq.dq = dq;
  pq.B = B;
  pq.H = H;
  pq.N = N;
  pq.d = d;
  pq.scale = scale;
  pq.causal = p.causal;
  pq.err = err;
  pq.wait_ns = p.wait_ns;
  FA_CUDA(fa::launch_backward_dq(pq, tq, tk, tv, tdo, stream));
  return FA_OK;
}

fa_status fa_forward_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int N, int d, float scale, int causal, float p_drop,
                             unsigned long long seed, unsigned offset, cudaStream_t stream) {
  FA_TRY(check_fwd_args(q, k, v, o, lse, B, H, N, d, scale));
  fa::DropoutParams drop;
  FA_TRY(make_dropout(p_drop, seed, offset, &drop));
  return forward_impl(q, k, v, o, lse, B, H, H, N, d, scale, causal, nullptr, stream, Varlen(),
                      drop);
}

fa_status fa_backward_dropout(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, float scale, int causal, float p_drop,
                              unsigned long long seed, unsigned offset, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  FA_TRY(check_bwd_args(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale));
  fa::DropoutParams drop;
  FA_TRY(make_dropout(p_drop, seed, offset, &drop));
  FA_TRY(check_ws(workspace, workspace_bytes, bwd_ws_bytes(B, H, N, d)));
  FA_TRY(fa_backward_preprocess(o, dO, B, H, N, d, workspace, workspace_bytes, stream));
  FA_TRY(backward_main_impl(q, k, v, dO, lse, dk, dv, B, H, H, N, d, scale, causal,
                            bwd_ws(workspace, B, H, N, d), nullptr, stream, Varlen(), drop));
  return fa_backward_dq_convert(dq, B, H, N, d, scale, workspace, workspace_bytes, stream);
}

size_t fa_blocksparse_workspace_size(int B, int H, int N, int d, int mask_heads) {
  if (B < 1 || H < 1 || N < 1 || d < 1 || mask_heads < 1) return 0;
  return lists_bytes(N, mask_heads) + bwd_ws_bytes(B, H, N, d);
}

fa_status fa_blocksparse_build_lists(const uint8_t* block_mask, int mask_heads, int N,
                                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (N < 1 || mask_heads < 1 || !block_mask) return FA_ERR_INVALID_ARG;
  if (num_tiles(N) > 8192) return FA_ERR_UNSUPPORTED;
  FA_TRY(check_ws(workspace, workspace_bytes, lists_bytes(N, mask_heads)));
  return build_lists(block_mask, mask_heads, N, workspace, stream);
}

fa_status fa_blocksparse_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int N, int d, float scale, int causal,
                                 const uint8_t* block_mask, int mask_heads, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
  FA_TRY(check_fwd_args(q, k, v, o, lse, B, H, N, d, scale));
  FA_TRY(check_mask(block_mask, mask_heads, H, N));
  FA_TRY(check_ws(workspace, workspace_bytes, lists_bytes(N, mask_heads)));
  FA_TRY(build_lists(block_mask, mask_heads, N, workspace, stream));
  const fa::TileLists L = lists_in(workspace, N, mask_heads);
  return forward_impl(q, k, v, o, lse, B, H, H, N, d, scale, causal, &L, stream);
}

fa_status fa_blocksparse_backward(const void* q, const void* k, const void* v, const void* o,
                                  const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                  int B, int H, int N, int d, float scale, int causal,
                                  const uint8_t* block_mask, int mask_heads, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
  FA_TRY(check_bwd_args(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale));
  FA_TRY(check_mask(block_mask, mask_heads, H, N));
  const size_t lb = lists_bytes(N, mask_heads);
  FA_TRY(check_ws(workspace, workspace_bytes, lb + bwd_ws_bytes(B, H, N, d)));
  FA_TRY(build_lists(block_mask, mask_heads, N, workspace, stream));
  const fa::TileLists L = lists_in(workspace, N, mask_heads);
  void* bws = static_cast<char*>(workspace) + lb;
  const size_t bws_bytes = workspace_bytes - lb;
  FA_TRY(fa_backward_preprocess(o, dO, B, H, N, d, bws, bws_bytes, stream));
  FA_TRY(backward_main_impl(q, k, v, dO, lse, dk, dv, B, H, H, N, d, scale, causal,
                            bwd_ws(bws, B, H, N, d), &L, stream));
  return fa_backward_dq_convert(dq, B, H, N, d, scale, bws, bws_bytes, stream);
}

fa_status fa_get_device_status(cudaStream_t stream) {
  fa_status st = FA_OK;
  int* w = status_word(&st);
  if (!w) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyAsync(&v, w, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return FA_ERR_CUDA;
  if (cudaMemsetAsync(w, 0, sizeof(int), stream) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  if (v == 0) return FA_OK;
  return v == FA_ERR_TIMEOUT ? FA_ERR_TIMEOUT : FA_ERR_CUDA;
}

fa_status fa_set_wait_limit_ns(unsigned long long ns) {
  g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns);
  return FA_OK;
}

fa_status fa_debug_wait_timeout(unsigned long long limit_ns, cudaStream_t stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return FA_ERR_INVALID_ARG;
  fa_status st = FA_OK;
  int* err = status_word(&st);
  if (!err) return st;
  FA_CUDA(fa::launch_wait_probe(err, limit_ns, stream));
  return FA_OK;
}

fa_status fa_debug_schedule(int N, int causal, const uint8_t* block_mask, int mask_heads,
                            void* workspace, size_t workspace_bytes, int* fwd_counts,
                            int* bwd_counts, int* fwd_lists, int* bwd_lists, cudaStream_t stream) {
  if (N < 1 || !fwd_counts || !bwd_counts || !fwd_lists || !bwd_lists) return FA_ERR_INVALID_ARG;
  if (num_tiles(N) > 8192) return FA_ERR_UNSUPPORTED;
  fa::TileLists L;
  int heads = 1;
  if (block_mask) {
    if (mask_heads < 1) return FA_ERR_INVALID_ARG;
    FA_TRY(check_ws(workspace, workspace_bytes, lists_bytes(N, mask_heads)));
    FA_TRY(build_lists(block_mask, mask_heads, N, workspace, stream));
    L = lists_in(workspace, N, mask_heads);
    heads = mask_heads;
  }
  FA_CUDA(fa::launch_schedule_export(N, causal, L, heads, fwd_counts, bwd_counts, fwd_lists,
                                     bwd_lists, stream));
  return FA_OK;
}

fa_status fa_debug_forward_config(const void* q, const void* k, const void* v, void* o,
                                  float* lse, int B, int H, int N, int d, float scale, int causal,
                                  int rows_per_cta, int key_tile, int kv_stages,
                                  cudaStream_t stream) {
  FA_TRY(check_fwd_args(q, k, v, o, lse, B, H, N, d, scale));
  if (!sweep_config_ok(d, rows_per_cta, key_tile, kv_stages)) return FA_ERR_UNSUPPORTED;
  fa_status st = FA_OK;
  int* err = status_word(&st);
  if (!err) return st;
  const int kbox = key_tile < kTile ? key_tile : kTile;
  CUtensorMap tq, tk, tv;
  if (!fa::make_tile_map(&tq, q, B * H, N, d) || !fa::make_tile_map(&tk, k, B * H, N, d, kbox) ||
      !fa::make_tile_map(&tv, v, B * H, N, d, kbox))
    return FA_ERR_CUDA;
  fa::FwdParams p;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Hkv = H;
  p.N = N;
  p.d = d;
  p.scale = scale;
  p.causal = causal ? 1 : 0;
  p.single_tile = rows_per_cta == 128 ? 1 : 0;
  p.err = err;
  p.wait_ns = wait_limit_ns();
  FA_CUDA(fa::launch_forward_config(p, tq, tk, tv, kv_stages, key_tile, stream));
  return FA_OK;
}

fa_status fa_debug_mma_probe(const void* a, const void* b, float* c, int mode, int n,
                             cudaStream_t stream) {
  if (mode < 0 || mode > 3) return FA_ERR_INVALID_ARG;
  if (mode == 0) n = 128;
  if (n != 64 && n != 128) return FA_ERR_UNSUPPORTED;
  FA_TRY(check_ptr16(a));
  FA_TRY(check_ptr16(b));
  FA_TRY(check_ptr16(c));
  fa_status st = FA_OK;
  int* err = status_word(&st);
  if (!err) return st;
  CUtensorMap ta, tb;
  if (!fa::make_tile_map(&ta, a, 1, 128, 128) || !fa::make_tile_map(&tb, b, 1, 128, n))
    return FA_ERR_CUDA;
  FA_CUDA(fa::launch_mma_probe(ta, tb, a, c, mode, n, err, wait_limit_ns(), stream));
  return FA_OK;
}

}  // extern "C"
