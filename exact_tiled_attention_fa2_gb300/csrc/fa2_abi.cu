// fa2_abi.cu -- the C ABI declared in include/fa2.h: argument checks, TMA
// tensor maps, the per-device status word, kernel dispatch and the
// host-buffer end-to-end entry point.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa2.h"
#include "fa2_common.cuh"
#include "fa2_decode.cuh"
#include "fa2_internal.h"

namespace fa2 {

// Written by kernels when a bounded wait gives up; one per device context.
__device__ uint32_t g_device_status;

TileGeometry tile_geometry(int d) {
  TileGeometry g;
  (void)d;   // the double-buffered kernel's tiles at every head dim
  g.q_rows = 128;
  g.kv_rows = 64;
  g.cta_rows = 128;
  return g;
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool supported = false;
  uint32_t* status = nullptr;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-device set-up: capability check and the status word's device address.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA2_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA2_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_devices[dev];
  if (!s.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FA2_ERR_CUDA;
    s.supported = (prop.major == 10 && prop.minor == 3);
    if (s.supported) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return FA2_ERR_CUDA;
      s.status = static_cast<uint32_t*>(addr);
      uint32_t zero = 0;
      if (cudaMemcpy(s.status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FA2_ERR_CUDA;
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return FA2_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    s.ready = true;
  }
  if (!s.supported) return FA2_ERR_UNSUPPORTED;
  *out = &s;
  return FA2_OK;
}

// Whether (batch, head) of a tensor with element strides st = {batch, head,
// row} can be addressed as one coordinate b*H + h with a single stride.
bool mergeable(long long heads, long long batch, const long long st[3]) {
  return heads == 1 || batch == 1 || st[0] == heads * st[1];
}

// View of a 16-bit tensor with element strides st = {batch, head, row}: 3-D
// (d, rows, heads*batch) when `merged` (see mergeable), else 4-D (d, rows,
// heads, batch); boxes of 64 columns x `box_rows` rows, 128-byte swizzle.
// Rows past `rows` read as zeros.  The stride of a dimension of size 1 never
// addresses anything and is replaced by a valid placeholder.
int encode_map_rows(CUtensorMap* m, const void* base, int d, long long rows, long long heads, long long batch,
                    const long long st[3], int box_rows, bool bf16, bool merged, int box_cols = 64,
                    CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const long long row_st = rows > 1 ? st[2] : d, head_st = heads > 1 ? st[1] : d, batch_st = batch > 1 ? st[0] : d;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads, (cuuint64_t)batch};
  cuuint64_t strides[3] = {(cuuint64_t)row_st * 2, (cuuint64_t)head_st * 2, (cuuint64_t)batch_st * 2};
  cuuint32_t box[4] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  cuuint32_t rank = 4;
  if (merged) {
    dims[2] = (cuuint64_t)(heads * batch);
    strides[1] = (cuuint64_t)(heads > 1 ? head_st : batch_st) * 2;
    rank = 3;
  }
  CUresult r = g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA2_OK : FA2_ERR_CUDA;
}

// Everything the forward tensor maps depend on.  Zero-filled before use so
// that whole-struct comparison is exact.
struct MapKey {
  int dev, dtype, d, merged;
  const void* ptr[4];        // q, k, v, o
  long long dims[4][3];      // rows, heads, batch of each
  long long strides[4][3];   // batch, head, row strides of each (elements)
};

// The tensor maps of the last forward (and, separately, decode) call on this
// host thread: repeated calls on the same buffers and shapes (the usual case
// in a loop) skip re-encoding them.
struct MapCache {
  bool valid = false;
  MapKey key;
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
};
thread_local MapCache t_maps;
thread_local MapCache t_decode_maps;
thread_local MapCache t_decode_tc_maps;
thread_local MapCache t_bwd_maps;

// K and V maps of the decode kernel: whole rows (d columns) x
// decode_block_rows(d) rows per box, no swizzle (rows land contiguously).
int cached_decode_maps(DecodeLaunchArgs& a, const MapKey& key) {
  MapCache& c = t_decode_maps;
  if (!(c.valid && std::memcmp(&c.key, &key, sizeof(MapKey)) == 0)) {
    const bool bf16 = key.dtype == FA2_BF16;
    CUtensorMap* maps[2] = {&c.tm_k, &c.tm_v};
    c.valid = false;
    for (int i = 0; i < 2; ++i) {
      if (encode_map_rows(maps[i], key.ptr[i + 1], key.d, key.dims[i + 1][0], key.dims[i + 1][1],
                          key.dims[i + 1][2], key.strides[i + 1], decode_block_rows(key.d), bf16, key.merged != 0,
                          key.d, CU_TENSOR_MAP_SWIZZLE_NONE))
        return FA2_ERR_CUDA;
    }
    std::memcpy(&c.key, &key, sizeof(MapKey));
    c.valid = true;
  }
  a.tm_k = c.tm_k;
  a.tm_v = c.tm_v;
  return FA2_OK;
}

// q, k, v and o maps with boxes of 64 columns x rows[t] rows (128-byte
// swizzle), cached per host thread in `c` (each cache serves one box geometry
// per head dim).
int cached_maps_rows(MapCache& c, LaunchArgs& a, const MapKey& key, const int rows[4]) {
  if (!(c.valid && std::memcmp(&c.key, &key, sizeof(MapKey)) == 0)) {
    const bool bf16 = key.dtype == FA2_BF16;
    CUtensorMap* maps[4] = {&c.tm_q, &c.tm_k, &c.tm_v, &c.tm_o};
    c.valid = false;
    for (int i = 0; i < 4; ++i) {
      if (encode_map_rows(maps[i], key.ptr[i], key.d, key.dims[i][0], key.dims[i][1], key.dims[i][2],
                          key.strides[i], rows[i], bf16, key.merged != 0))
        return FA2_ERR_CUDA;
    }
    std::memcpy(&c.key, &key, sizeof(MapKey));
    c.valid = true;
  }
  a.tm_q = c.tm_q;
  a.tm_k = c.tm_k;
  a.tm_v = c.tm_v;
  a.tm_o = c.tm_o;
  return FA2_OK;
}

// The forward kernel's maps: query tiles, key/value tiles (tile_geometry) and
// o boxes of one warp's 32 rows.
int cached_maps(LaunchArgs& a, const MapKey& key) {
  const TileGeometry g = tile_geometry(key.d);
  const int rows[4] = {g.q_rows, g.kv_rows, g.kv_rows, 32};
  return cached_maps_rows(t_maps, a, key, rows);
}

// Maps of the tensor-core decode path: the forward kernel's geometry (o is not
// stored through in split-key mode, but every map the kernel prefetches is valid).
int cached_decode_tc_maps(LaunchArgs& a, const MapKey& key) {
  const int rows[4] = {128, 64, 64, 32};
  return cached_maps_rows(t_decode_tc_maps, a, key, rows);
}

// The backward kernels' q, k and v maps: 128-row key tiles; query tiles of
// 128 rows (d = 128) or 64 rows (d = 64, 256).
int bwd_query_rows(int d) { return d == 128 ? 128 : 64; }
int cached_bwd_maps(LaunchArgs& a, const MapKey& key) {
  const int rows[4] = {bwd_query_rows(key.d), 128, 128, 32};
  return cached_maps_rows(t_bwd_maps, a, key, rows);
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// Checks that need no CUDA call.  Sizes in elements.
int check_shape(int B, int H, int N, int d, float scale, int causal, int dtype) {
  if (dtype != FA2_FP16 && dtype != FA2_BF16) return FA2_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return FA2_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA2_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA2_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA2_ERR_UNSUPPORTED;
  // one block per (head, query tile) in a 1-D grid
  if ((long long)B * (long long)H * (long long)((N + 127) / 128) > INT_MAX) return FA2_ERR_UNSUPPORTED;
  return FA2_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace fa2

using namespace fa2;

namespace fa2 {
namespace {

// Byte range [base, base + span) a strided 16-bit tensor (or float32 when
// elem == 4) can touch: dims = {batch, heads, rows}, strides in elements,
// `inner` contiguous elements per row.
struct Extent {
  const void* base;
  size_t bytes;
};

Extent extent(const void* base, const long long dims[3], const long long st[3], long long inner, int elem) {
  long long last = inner - 1;
  for (int i = 0; i < 3; ++i)
    if (dims[i] > 1) last += (dims[i] - 1) * st[i];
  return Extent{base, (size_t)(last + 1) * (size_t)elem};
}

bool overlap(const Extent& a, const Extent& b) { return ranges_overlap(a.base, a.bytes, b.base, b.bytes); }

constexpr long long kMaxStride = 1ll << 39;  // elements: 16-bit strides stay below the TMA limit of 2^40 bytes

// 0, or the status for a stride of a dimension of size n.
int check_stride(long long n, long long st, bool tma) {
  if (n <= 1) return FA2_OK;
  if (st <= 0 || st >= kMaxStride) return FA2_ERR_INVALID_ARG;
  if (tma && (st & 7)) return FA2_ERR_MISALIGNED;
  return FA2_OK;
}

// A batch whose (batch, head) strides merge in every tensor (batch stride =
// H x head stride, as in contiguous [B,H,N,d]) runs as one batch of B*H
// heads: the kernels then need no division to find a CTA's batch.
fa2_fwd_params fold_batches(const fa2_fwd_params& a_in) {
  fa2_fwd_params a = a_in;
  const bool packed = a.cu_seqlens_q != nullptr || a.cu_seqlens_k != nullptr;
  if (!packed && a.batch > 1 && a.heads > 1) {
    const int64_t* st[4] = {a.q_strides, a.k_strides, a.v_strides, a.o_strides};
    bool fold = a.lse_strides[0] == (int64_t)a.heads * a.lse_strides[1];
    for (const int64_t* s : st) fold = fold && s[0] == (int64_t)a.heads * s[1];
    if (fold && (long long)a.batch * a.heads <= INT_MAX) {
      a.heads *= a.batch;
      a.batch = 1;
    }
  }
  return a;
}

// Validated arguments turned into kernel parameters and map descriptions.
struct Prepared {
  KernelParams p;
  MapKey key;            // q, k, v: pointers, dims, strides, rank
  long long q_st[3];     // q strides (the decode kernel reads q directly)
  bool band;             // a row's first visible key depends on the row
};

// Checks every argument (no CUDA call before they pass), then fills `out`;
// `units_rows` is the query rows one CTA covers (sizes KernelParams.units).
// `scratch` (optional): a further buffer the launch writes, which must overlap
// none of the tensors.
int prepare(const fa2_fwd_params& a, int units_rows, Prepared& out, const Extent* scratch = nullptr) {
  if (a.dtype != FA2_FP16 && a.dtype != FA2_BF16) return FA2_ERR_INVALID_ARG;
  if (a.batch < 1 || a.heads < 1 || a.seqlen_q < 1) return FA2_ERR_INVALID_ARG;
  if (!std::isfinite(a.scale)) return FA2_ERR_INVALID_ARG;
  if (a.window_left < -1 || a.window_right < -1 || a.prefix_len < 0) return FA2_ERR_INVALID_ARG;
  const int d = a.head_dim;
  if (d != 64 && d != 128 && d != 256) return FA2_ERR_UNSUPPORTED;
  const bool packed = a.cu_seqlens_q != nullptr || a.cu_seqlens_k != nullptr;
  if (packed && !(a.cu_seqlens_q && a.cu_seqlens_k)) return FA2_ERR_INVALID_ARG;
  if (packed ? (a.total_q < 1 || a.total_k < 1) : a.seqlen_k < 1) return FA2_ERR_INVALID_ARG;
  if (!a.q || !a.k || !a.v || !a.o || !a.lse) return FA2_ERR_INVALID_ARG;
  if (misaligned(a.q) || misaligned(a.k) || misaligned(a.v) || misaligned(a.o)) return FA2_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(a.lse) & 3u) return FA2_ERR_MISALIGNED;
  if (packed && ((reinterpret_cast<uintptr_t>(a.cu_seqlens_q) | reinterpret_cast<uintptr_t>(a.cu_seqlens_k)) & 3u))
    return FA2_ERR_MISALIGNED;
  const long long units = ((long long)a.seqlen_q + units_rows - 1) / units_rows;
  if ((long long)a.batch * a.heads * units > INT_MAX) return FA2_ERR_UNSUPPORTED;

  // tensor batch dimension (1 when packed: sequences are rows) and row counts
  const long long tb = packed ? 1 : a.batch;
  const long long rows_q = packed ? a.total_q : a.seqlen_q;
  const long long rows_k = packed ? a.total_k : a.seqlen_k;
  const long long dq[3] = {tb, a.heads, rows_q}, dk[3] = {tb, a.heads, rows_k};
  long long st_in[3][3];
  const int64_t* st_src[3] = {a.q_strides, a.k_strides, a.v_strides};
  for (int t = 0; t < 3; ++t)
    for (int i = 0; i < 3; ++i) st_in[t][i] = (long long)st_src[t][i];
  for (int t = 0; t < 3; ++t) {
    const long long* dims = t == 0 ? dq : dk;
    for (int i = 0; i < 3; ++i) {
      const int rc = check_stride(dims[i], st_in[t][i], true);
      if (rc) return rc;
    }
  }
  for (int i = 0; i < 3; ++i) {
    const int rc = check_stride(dq[i], a.o_strides[i], true);
    if (rc) return rc;
  }
  const long long lse_st[3] = {packed ? 0 : (long long)a.lse_strides[0], (long long)a.lse_strides[1], 1};
  for (int i = 0; i < 2; ++i)
    if (dq[i] > 1 && (lse_st[i] < 0 || lse_st[i] >= kMaxStride)) return FA2_ERR_INVALID_ARG;
  // o and lse overlap nothing they are not
  const long long o_st[3] = {(long long)a.o_strides[0], (long long)a.o_strides[1], (long long)a.o_strides[2]};
  const Extent e_o = extent(a.o, dq, o_st, d, 2), e_l = extent(a.lse, dq, lse_st, 1, 4);
  const Extent ins[3] = {extent(a.q, dq, st_in[0], d, 2), extent(a.k, dk, st_in[1], d, 2),
                         extent(a.v, dk, st_in[2], d, 2)};
  if (overlap(e_o, e_l)) return FA2_ERR_INVALID_ARG;
  for (const Extent& in : ins)
    if (overlap(e_o, in) || overlap(e_l, in)) return FA2_ERR_INVALID_ARG;
  if (scratch) {
    if (overlap(*scratch, e_o) || overlap(*scratch, e_l)) return FA2_ERR_INVALID_ARG;
    for (const Extent& in : ins)
      if (overlap(*scratch, in)) return FA2_ERR_INVALID_ARG;
  }

  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc) return rc;
  MapKey& key = out.key;
  std::memset(&key, 0, sizeof(key));
  if (cudaGetDevice(&key.dev) != cudaSuccess) return FA2_ERR_CUDA;
  key.dtype = a.dtype;
  key.d = d;
  const void* ptrs[4] = {a.q, a.k, a.v, a.o};
  for (int t = 0; t < 4; ++t) {
    const long long* dims = (t == 0 || t == 3) ? dq : dk;
    key.ptr[t] = ptrs[t];
    key.dims[t][0] = dims[2];  // rows, heads, batch
    key.dims[t][1] = dims[1];
    key.dims[t][2] = dims[0];
    for (int i = 0; i < 3; ++i) key.strides[t][i] = t < 3 ? st_in[t][i] : o_st[i];
  }
  // one map rank for every tensor: merge (batch, head) only when q, k, v and
  // o all allow it (the backward's dout shares o's strides)
  key.merged = 1;
  for (int t = 0; t < 4; ++t)
    if (!mergeable(a.heads, tb, key.strides[t])) key.merged = 0;
  for (int i = 0; i < 3; ++i) out.q_st[i] = st_in[0][i];
  KernelParams& p = out.p;
  std::memset(&p, 0, sizeof(p));
  p.o = a.o;
  p.lse = a.lse;
  p.status = ds->status;
  p.cu_q = packed ? a.cu_seqlens_q : nullptr;
  p.cu_k = packed ? a.cu_seqlens_k : nullptr;
  p.o_bs = packed ? 0 : a.o_strides[0];
  p.o_hs = a.o_strides[1];
  p.o_rs = a.o_strides[2];
  p.l_bs = lse_st[0];
  p.l_hs = lse_st[1];
  p.n_q = a.seqlen_q;
  p.n_k = packed ? a.total_k : a.seqlen_k;
  p.total_q = (int)rows_q;
  p.total_k = (int)rows_k;
  p.heads = a.heads;
  p.merged_bh = key.merged;
  p.tma_o = packed ? 0 : 1;   // packed: a box would spill into the next sequence's rows
  p.bh = a.batch * a.heads;
  p.units = (int)units;
  p.window_left = a.window_left;
  p.window_right = a.window_right;
  p.prefix = a.prefix_len;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.scale_log2_mag = std::fmax(std::fabs(p.scale_log2), FLT_MIN);
  p.qk_negate = p.scale_log2 < 0.f ? kIdescNegateA : 0u;
  out.band = a.window_left >= 0 || a.prefix_len > 0;
  return FA2_OK;
}

// Units per head of a packed batch's grid when each CTA finds its own tile
// from the offsets (kernels' packed_unit; at most kPackedScanSeqs sequences),
// or 0 for the plain grid of `units_each` units per (sequence, head).
// Sequences whose rows do not overlap hold at most (total + (rows - 1) * B) /
// rows whole or partial tiles of `rows` rows; the smaller grid wins.
long long packed_grid_units(const fa2_fwd_params& a, long long total, int rows, long long units_each) {
  if (!a.cu_seqlens_q || a.batch > kPackedScanSeqs) return 0;
  const long long u = (total + (long long)(rows - 1) * a.batch) / rows;
  return u < units_each * a.batch ? u : 0;
}

// Validates the general forward arguments (no CUDA call before they pass),
// then launches the tiled kernel for the head dim.
int forward(const fa2_fwd_params& a_in, cudaStream_t stream) {
  const fa2_fwd_params a = fold_batches(a_in);
  Prepared pr;
  const int rows = tile_geometry(a.head_dim).cta_rows;
  int rc = prepare(a, rows, pr);
  if (rc) return rc;
  pr.p.packed_units = (int)packed_grid_units(a, a.total_q, rows, pr.p.units);   // <= the plain grid
  LaunchArgs la;
  std::memset(&la, 0, sizeof(la));
  rc = cached_maps(la, pr.key);
  if (rc) return rc;
  la.p = pr.p;
  la.bf16 = a.dtype == FA2_BF16;
  la.band = pr.band;
  la.stream = stream;
  int e = 0;
  switch (a.head_dim) {
    case 64: e = launch_fwd_d64(la); break;
    case 128: e = launch_fwd_d128(la); break;
    default: e = launch_fwd_d256(la); break;
  }
  return e == 0 ? FA2_OK : FA2_ERR_CUDA;
}

// Key splits of the decode path: enough CTAs for two on each of the 152 SMs
// of a GB300 (independent of the device, so the workspace size is too), no
// split shorter than kDecodeMinChunk keys, chunks a multiple of a stage.
constexpr long long kDecodeTargetCtas = 2 * 152;
constexpr long long kDecodeMinChunk = 256;
// From this many query rows on the chunks run on the tensor cores (the tiled
// kernel in split-key mode); fewer rows, and d = 256, stay on the CUDA-core
// decode kernel.  Measured: at d = 128 the tensor-core path is 2-8 % faster
// already for one row; at d = 64 one row is 8 % faster on CUDA cores.
constexpr int decode_tc_min_rows(int d) { return d == 128 ? 1 : d == 64 ? 2 : 1 << 30; }

struct DecodePlan {
  int splits, chunk, base;
  size_t ws_o_bytes, ws_ml_bytes;
};

// 0, or a status: N_q <= FA2_DECODE_MAX_Q, plus the plan for these sizes.
int decode_plan(const fa2_fwd_params& a, DecodePlan& out) {
  if (a.seqlen_q < 1 || a.seqlen_q > FA2_DECODE_MAX_Q) return FA2_ERR_UNSUPPORTED;
  if (a.seqlen_k < 1 || a.batch < 1 || a.heads < 1) return FA2_ERR_INVALID_ARG;
  if (a.head_dim != 64 && a.head_dim != 128 && a.head_dim != 256) return FA2_ERR_UNSUPPORTED;
  const long long bh = (long long)a.batch * a.heads;
  const long long nk = a.seqlen_k;
  const long long block = decode_block_rows(a.head_dim);
  // Keys before the first one query row 0 sees (a bounded left window, no
  // prefix) are seen by no row: the chunks start at that key, rounded down to
  // a stage.  Packed sequences differ in length: their chunks start at 0.
  long long base = 0;
  const bool packed = a.cu_seqlens_q != nullptr;
  if (!packed && a.window_left >= 0 && a.prefix_len <= 0) {
    const long long first = nk - a.seqlen_q - a.window_left;
    if (first > 0) base = (first < nk ? first : nk - 1) / block * block;
  }
  const long long span = nk - base;
  long long splits = kDecodeTargetCtas / bh;
  const long long useful = (span + kDecodeMinChunk - 1) / kDecodeMinChunk;
  if (splits > useful) splits = useful;
  if (splits < 1) splits = 1;
  long long chunk = (span + splits - 1) / splits;
  chunk = (chunk + block - 1) / block * block;
  splits = (span + chunk - 1) / chunk;
  if (bh * splits > INT_MAX || bh * a.seqlen_q > INT_MAX) return FA2_ERR_UNSUPPORTED;
  out.splits = (int)splits;
  out.chunk = (int)chunk;
  out.base = (int)base;
  const size_t slots = (size_t)bh * (size_t)a.seqlen_q * (size_t)splits;
  out.ws_o_bytes = align256(slots * (size_t)a.head_dim * 4);
  out.ws_ml_bytes = align256(slots * 2 * 4);
  return FA2_OK;
}

int decode(const fa2_fwd_params& a_in, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const fa2_fwd_params a = fold_batches(a_in);
  DecodePlan plan;
  int rc = decode_plan(a, plan);
  if (rc) return rc;
  if (!workspace) return FA2_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA2_ERR_MISALIGNED;
  if (workspace_bytes < plan.ws_o_bytes + plan.ws_ml_bytes) return FA2_ERR_INVALID_ARG;
  // the workspace is written by the kernels: it must overlap none of the tensors
  const Extent ew{workspace, plan.ws_o_bytes + plan.ws_ml_bytes};
  Prepared pr;
  rc = prepare(a, FA2_DECODE_MAX_Q, pr, &ew);
  if (rc) return rc;
  const bool packed = a.cu_seqlens_q != nullptr;
  if (a.seqlen_q >= decode_tc_min_rows(a.head_dim)) {
    // one query tile (N_q <= 8) per (b, h) or packed sequence, split into the
    // plan's key chunks (a multiple of the kernel's 64-row key tile)
    LaunchArgs tl;
    std::memset(&tl, 0, sizeof(tl));
    rc = cached_decode_tc_maps(tl, pr.key);
    if (rc) return rc;
    tl.p = pr.p;
    tl.p.tma_o = 0;
    tl.p.units = plan.splits;
    tl.p.splits = plan.splits;
    tl.p.split_chunk = plan.chunk;
    tl.p.split_base = plan.base;
    tl.p.ws_o = static_cast<float*>(workspace);
    tl.p.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.ws_o_bytes);
    tl.bf16 = a.dtype == FA2_BF16;
    tl.band = pr.band;
    tl.stream = stream;
    const int e = a.head_dim == 64 ? launch_decode_tc_d64(tl) : launch_decode_tc_d128(tl);
    return e == 0 ? FA2_OK : FA2_ERR_CUDA;
  }
  DecodeLaunchArgs la;
  std::memset(&la, 0, sizeof(la));
  rc = cached_decode_maps(la, pr.key);
  if (rc) return rc;
  la.p.q = a.q;
  la.p.q_bs = packed ? 0 : pr.q_st[0];
  la.p.q_hs = pr.q_st[1];
  la.p.q_rs = pr.q_st[2];
  la.p.ws_o = static_cast<float*>(workspace);
  la.p.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.ws_o_bytes);
  la.p.splits = plan.splits;
  la.p.chunk = plan.chunk;
  la.p.base = plan.base;
  la.p.f = pr.p;
  la.p.f.n_k = a.seqlen_k;   // packed: the longest sequence's key count the plan covers
  la.bf16 = a.dtype == FA2_BF16;
  la.stream = stream;
  // d = 128 always takes the tensor-core path above
  const int e = a.head_dim == 64 ? launch_decode_d64(la) : launch_decode_d256(la);
  return e == 0 ? FA2_OK : FA2_ERR_CUDA;
}

}  // namespace
}  // namespace fa2

extern "C" size_t fa2_fwd_params_size(void) { return sizeof(fa2_fwd_params); }

extern "C" int fa2_fwd_ex(const fa2_fwd_params* params, void* stream) {
  if (!params) return FA2_ERR_INVALID_ARG;
  return forward(*params, static_cast<cudaStream_t>(stream));
}

extern "C" size_t fa2_decode_workspace_bytes(const fa2_fwd_params* params) {
  if (!params) return 0;
  DecodePlan plan;
  if (decode_plan(fold_batches(*params), plan)) return 0;
  return plan.ws_o_bytes + plan.ws_ml_bytes;
}

extern "C" int fa2_decode(const fa2_fwd_params* params, void* workspace, size_t workspace_bytes, void* stream) {
  if (!params) return FA2_ERR_INVALID_ARG;
  return decode(*params, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" int fa2_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                       int d, float scale, int causal, int dtype, void* stream) {
  int rc = check_shape(B, H, N, d, scale, causal, dtype);
  if (rc) return rc;
  if (!q || !k || !v || !o || !lse) return FA2_ERR_INVALID_ARG;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o) || misaligned(lse)) return FA2_ERR_MISALIGNED;
  fa2_fwd_params a;
  std::memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.batch = B;
  a.heads = H;
  a.seqlen_q = N;
  a.seqlen_k = N;
  a.head_dim = d;
  a.dtype = dtype;
  a.scale = scale;
  a.window_left = -1;
  a.window_right = causal ? 0 : -1;
  a.prefix_len = 0;
  const long long row = d, head = (long long)N * d, batch = (long long)H * N * d;
  int64_t* st[4] = {a.q_strides, a.k_strides, a.v_strides, a.o_strides};
  for (int64_t* s : st) {
    s[0] = batch;
    s[1] = head;
    s[2] = row;
  }
  a.lse_strides[0] = (long long)H * N;
  a.lse_strides[1] = N;
  return forward(a, static_cast<cudaStream_t>(stream));
}

extern "C" size_t fa2_fwd_host_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  const size_t elems = (size_t)B * H * (size_t)N * d;
  return 4 * align256(elems * 2) + align256((size_t)B * H * (size_t)N * 4);
}

namespace fa2 {
namespace {

// Checks shared by the host-buffer entry points.
int check_host_args(const void* q_host, const void* k_host, const void* v_host, const void* o_host,
                    const float* lse_host, const void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                    float scale, int causal, int dtype) {
  int rc = check_shape(B, H, N, d, scale, causal, dtype);
  if (rc) return rc;
  if (!q_host || !k_host || !v_host || !o_host || !lse_host || !workspace) return FA2_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA2_ERR_MISALIGNED;
  if (workspace_bytes < fa2_fwd_host_workspace_bytes(B, H, N, d)) return FA2_ERR_INVALID_ARG;
  return FA2_OK;
}

// Whole problem in one pass on `stream`: copy in, forward, copy out,
// synchronise.  Every return after the first queued copy -- an error
// included -- first synchronises `stream`, so no copy into the workspace or
// the caller's host buffers is still in flight when the call returns.
int host_forward_serial(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                        void* workspace, int B, int H, int N, int d, float scale, int causal, int dtype,
                        void* stream) {
  const size_t elems = (size_t)B * H * (size_t)N * d;
  const size_t tb = elems * 2, lb = (size_t)B * H * (size_t)N * 4;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  void* qd = w;
  void* kd = w + align256(tb);
  void* vd = w + 2 * align256(tb);
  void* od = w + 3 * align256(tb);
  float* ld = reinterpret_cast<float*>(w + 4 * align256(tb));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto drained = [&](int status) {
    cudaStreamSynchronize(s);
    return status;
  };
  if (cudaMemcpyAsync(qd, q_host, tb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(kd, k_host, tb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(vd, v_host, tb, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return drained(FA2_ERR_CUDA);
  int rc = fa2_fwd(qd, kd, vd, od, ld, B, H, N, d, scale, causal, dtype, stream);
  if (rc) return drained(rc);
  if (cudaMemcpyAsync(o_host, od, tb, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(lse_host, ld, lb, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return drained(FA2_ERR_CUDA);
  return fa2_get_device_status(stream, nullptr);
}

// Library-owned copy streams and events of one device for the pipelined host
// path, created on first use and kept until exit.  The mutex serialises
// pipelined calls on the device (they share the streams and events).
constexpr int kMaxChunks = 8;
constexpr size_t kPipelineMinBytes = (size_t)48 << 20;

struct CopyEngines {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t entry = nullptr, in_done[kMaxChunks], fwd_done[kMaxChunks], out_done[kMaxChunks];
  std::mutex busy;
};
CopyEngines g_copy[kMaxDevices];

int copy_engines(CopyEngines** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA2_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA2_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  CopyEngines& c = g_copy[dev];
  if (!c.ready) {
    const unsigned f = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.entry, f) != cudaSuccess)
      return FA2_ERR_CUDA;
    for (int i = 0; i < kMaxChunks; ++i) {
      if (cudaEventCreateWithFlags(&c.in_done[i], f) != cudaSuccess ||
          cudaEventCreateWithFlags(&c.fwd_done[i], f) != cudaSuccess ||
          cudaEventCreateWithFlags(&c.out_done[i], f) != cudaSuccess)
        return FA2_ERR_CUDA;
    }
    c.ready = true;
  }
  *out = &c;
  return FA2_OK;
}

// The (b,h) slices are independent, so the problem is cut into up to
// kMaxChunks groups of heads: the copy-in of group c+1 (one stream) and the
// copy-out of group c-1 (another) run while the forward pass of group c runs
// on `stream`.
int host_forward_pipelined(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                           float* lse_host, void* workspace, int B, int H, int N, int d, float scale, int causal,
                           int dtype, void* stream) {
  const int bh = B * H;
  const size_t head_elems = (size_t)N * d;
  const size_t tb = (size_t)bh * head_elems * 2;
  if (3 * tb < kPipelineMinBytes || bh < 2)
    return host_forward_serial(q_host, k_host, v_host, o_host, lse_host, workspace, B, H, N, d, scale, causal,
                               dtype, stream);
  CopyEngines* ce = nullptr;
  int rc = copy_engines(&ce);
  if (rc) return rc;
  std::lock_guard<std::mutex> busy(ce->busy);
  const int chunks = bh < kMaxChunks ? bh : kMaxChunks;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  uint8_t* qd = w;
  uint8_t* kd = w + align256(tb);
  uint8_t* vd = w + 2 * align256(tb);
  uint8_t* od = w + 3 * align256(tb);
  float* ld = reinterpret_cast<float*>(w + 4 * align256(tb));
  const uint8_t* qh = static_cast<const uint8_t*>(q_host);
  const uint8_t* kh = static_cast<const uint8_t*>(k_host);
  const uint8_t* vh = static_cast<const uint8_t*>(v_host);
  uint8_t* oh = static_cast<uint8_t*>(o_host);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool ok = cudaEventRecord(ce->entry, s) == cudaSuccess &&
            cudaStreamWaitEvent(ce->h2d, ce->entry, 0) == cudaSuccess;
  // copy-in of every group, in order, on the copy-in stream
  for (int c = 0; c < chunks && ok; ++c) {
    const int h0 = (int)((long long)bh * c / chunks), h1 = (int)((long long)bh * (c + 1) / chunks);
    const size_t off = (size_t)h0 * head_elems * 2, bytes = (size_t)(h1 - h0) * head_elems * 2;
    ok = cudaMemcpyAsync(qd + off, qh + off, bytes, cudaMemcpyHostToDevice, ce->h2d) == cudaSuccess &&
         cudaMemcpyAsync(kd + off, kh + off, bytes, cudaMemcpyHostToDevice, ce->h2d) == cudaSuccess &&
         cudaMemcpyAsync(vd + off, vh + off, bytes, cudaMemcpyHostToDevice, ce->h2d) == cudaSuccess &&
         cudaEventRecord(ce->in_done[c], ce->h2d) == cudaSuccess;
  }
  // forward of each group once its inputs landed; copy-out once it finished
  for (int c = 0; c < chunks && ok; ++c) {
    const int h0 = (int)((long long)bh * c / chunks), h1 = (int)((long long)bh * (c + 1) / chunks);
    const size_t off = (size_t)h0 * head_elems * 2, bytes = (size_t)(h1 - h0) * head_elems * 2;
    ok = cudaStreamWaitEvent(s, ce->in_done[c], 0) == cudaSuccess;
    if (!ok) break;
    rc = fa2_fwd(qd + off, kd + off, vd + off, od + off, ld + (size_t)h0 * N, 1, h1 - h0, N, d, scale, causal,
                 dtype, stream);
    if (rc) break;
    ok = cudaEventRecord(ce->fwd_done[c], s) == cudaSuccess &&
         cudaStreamWaitEvent(ce->d2h, ce->fwd_done[c], 0) == cudaSuccess &&
         cudaMemcpyAsync(oh + off, od + off, bytes, cudaMemcpyDeviceToHost, ce->d2h) == cudaSuccess &&
         cudaMemcpyAsync(lse_host + (size_t)h0 * N, ld + (size_t)h0 * N, (size_t)(h1 - h0) * N * 4,
                         cudaMemcpyDeviceToHost, ce->d2h) == cudaSuccess &&
         cudaEventRecord(ce->out_done[c], ce->d2h) == cudaSuccess;
  }
  if (ok && rc == FA2_OK) ok = cudaStreamWaitEvent(s, ce->out_done[chunks - 1], 0) == cudaSuccess;
  // whatever happened, nothing of this call may still be in flight on return
  const bool drained = cudaStreamSynchronize(ce->h2d) == cudaSuccess && cudaStreamSynchronize(ce->d2h) == cudaSuccess;
  if (rc) return rc;
  if (!ok || !drained) return FA2_ERR_CUDA;
  return fa2_get_device_status(stream, nullptr);
}

}  // namespace
}  // namespace fa2

extern "C" int fa2_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                            float* lse_host, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                            float scale, int causal, int dtype, void* stream) {
  int rc = check_host_args(q_host, k_host, v_host, o_host, lse_host, workspace, workspace_bytes, B, H, N, d, scale,
                           causal, dtype);
  if (rc) return rc;
  return host_forward_pipelined(q_host, k_host, v_host, o_host, lse_host, workspace, B, H, N, d, scale, causal,
                                dtype, stream);
}

namespace fa2 {

// Device staging area of fa2_fwd_host_noalloc: a fixed-size array in the
// module's global memory, so that entry point never allocates.  Host code
// must not use the symbol as an address; it looks up the device address once
// per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[FA2_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mutex;
void* g_noalloc_address[kMaxDevices];

// Device address of g_noalloc_scratch on the current device (looked up on
// first use, with that device current).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA2_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA2_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_address[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FA2_ERR_CUDA;
    g_noalloc_address[dev] = p;
  }
  *out = g_noalloc_address[dev];
  return FA2_OK;
}

}  // namespace
}  // namespace fa2

extern "C" int fa2_fwd_host_noalloc(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                                    float* lse_host, int B, int H, int N, int d, float scale, int causal,
                                    int dtype, void* stream) {
  int rc = check_shape(B, H, N, d, scale, causal, dtype);
  if (rc) return rc;
  if (!q_host || !k_host || !v_host || !o_host || !lse_host) return FA2_ERR_INVALID_ARG;
  if (fa2_fwd_host_workspace_bytes(B, H, N, d) > FA2_NOALLOC_SCRATCH_BYTES) return FA2_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  return host_forward_serial(q_host, k_host, v_host, o_host, lse_host, scratch, B, H, N, d, scale, causal, dtype,
                             stream);
}

namespace fa2 {

// One thread waits, through the kernels' bounded-wait helper, on an mbarrier
// that nothing ever arrives on; the wait expires after limit_ns and records
// kSiteSelfTest in the status word, and the kernel returns normally.
__global__ void selftest_wait_timeout_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  wait_or_abort_for(b, 0, &abort_flag, status, kSiteSelfTest, limit_ns);
}

}  // namespace fa2

namespace fa2 {
namespace {

// fp32 (d, rows, B*H) view of the dQ accumulator; boxes of 32 columns x 32
// rows (one warp's rows and a 128-byte column block), 128-byte swizzle, for
// TMA reduce-add.  Rows past `rows` are clipped.
int encode_dq_accum_map(CUtensorMap* m, void* base, long long slices, long long rows, int d) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)slices};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)rows * (cuuint64_t)d * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA2_OK : FA2_ERR_CUDA;
}

struct BwdPlan {
  long long slices, rows_q;   // (tensor batch x heads) slices and query rows per slice
  int num_k_tiles;
  size_t accum_bytes, delta_bytes;
};

int bwd_plan(const fa2_fwd_params& a, BwdPlan& out) {
  if (a.head_dim != 64 && a.head_dim != 128 && a.head_dim != 256) return FA2_ERR_UNSUPPORTED;
  if (a.batch < 1 || a.heads < 1 || a.seqlen_q < 1 || a.seqlen_k < 1) return FA2_ERR_INVALID_ARG;
  const bool packed = a.cu_seqlens_q != nullptr;
  if (packed && a.total_q < 1) return FA2_ERR_INVALID_ARG;
  out.slices = (long long)(packed ? 1 : a.batch) * a.heads;
  out.rows_q = packed ? a.total_q : a.seqlen_q;
  const long long tiles = ((long long)a.seqlen_k + 127) / 128;
  // one CTA per key tile (d = 256: per key tile and half of d) in a 1-D grid
  if ((long long)a.batch * a.heads * tiles * (a.head_dim == 256 ? 2 : 1) > INT_MAX) return FA2_ERR_UNSUPPORTED;
  out.num_k_tiles = (int)tiles;
  const size_t rows = (size_t)out.slices * (size_t)out.rows_q;
  out.accum_bytes = align256(rows * (size_t)a.head_dim * 4);
  out.delta_bytes = align256(rows * 4);
  return FA2_OK;
}

int backward(const fa2_bwd_params& bp, cudaStream_t stream) {
  fa2_bwd_params b = bp;
  b.fwd = fold_batches(bp.fwd);
  const fa2_fwd_params& a = b.fwd;
  BwdPlan plan;
  int rc = bwd_plan(a, plan);
  if (rc) return rc;
  if (!b.dout || !b.dq || !b.dk || !b.dv || !b.workspace) return FA2_ERR_INVALID_ARG;
  if (misaligned(b.dout) || misaligned(b.dq) || misaligned(b.dk) || misaligned(b.dv)) return FA2_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(b.workspace) & 255u) return FA2_ERR_MISALIGNED;
  if (b.workspace_bytes < plan.accum_bytes + plan.delta_bytes) return FA2_ERR_INVALID_ARG;
  // byte ranges: every written buffer overlaps no input and no other output
  const bool packed = a.cu_seqlens_q != nullptr || a.cu_seqlens_k != nullptr;
  const long long tb = packed ? 1 : a.batch;
  const long long dq_dims[3] = {tb, a.heads, packed ? a.total_q : a.seqlen_q};
  const long long dk_dims[3] = {tb, a.heads, packed ? a.total_k : a.seqlen_k};
  long long st[4][3];
  const int64_t* src[4] = {a.q_strides, a.k_strides, a.v_strides, a.o_strides};
  for (int t = 0; t < 4; ++t)
    for (int i = 0; i < 3; ++i) st[t][i] = (long long)src[t][i];
  for (int i = 0; i < 3; ++i) {   // the stride checks prepare() repeats, needed here for the extents
    if (check_stride(dq_dims[i], st[0][i], true) || check_stride(dk_dims[i], st[1][i], true) ||
        check_stride(dk_dims[i], st[2][i], true) || check_stride(dq_dims[i], st[3][i], true))
      return FA2_ERR_INVALID_ARG;
  }
  const long long l_st[3] = {packed ? 0 : (long long)a.lse_strides[0], (long long)a.lse_strides[1], 1};
  const int d = a.head_dim;
  const Extent outs[4] = {extent(b.dq, dq_dims, st[0], d, 2), extent(b.dk, dk_dims, st[1], d, 2),
                          extent(b.dv, dk_dims, st[2], d, 2),
                          Extent{b.workspace, plan.accum_bytes + plan.delta_bytes}};
  const Extent ins[6] = {extent(a.q, dq_dims, st[0], d, 2),   extent(a.k, dk_dims, st[1], d, 2),
                         extent(a.v, dk_dims, st[2], d, 2),   extent(a.o, dq_dims, st[3], d, 2),
                         extent(a.lse, dq_dims, l_st, 1, 4), extent(b.dout, dq_dims, st[3], d, 2)};
  for (int i = 0; i < 4; ++i) {
    for (const Extent& in : ins)
      if (overlap(outs[i], in)) return FA2_ERR_INVALID_ARG;
    for (int j = i + 1; j < 4; ++j)
      if (overlap(outs[i], outs[j])) return FA2_ERR_INVALID_ARG;
  }
  Prepared pr;
  rc = prepare(a, 128, pr);
  if (rc) return rc;
  BwdLaunchArgs la;
  std::memset(&la, 0, sizeof(la));
  LaunchArgs fl;
  std::memset(&fl, 0, sizeof(fl));
  rc = cached_bwd_maps(fl, pr.key);
  if (rc) return rc;
  la.tm_q = fl.tm_q;
  la.tm_k = fl.tm_k;
  la.tm_v = fl.tm_v;
  const bool bf16 = a.dtype == FA2_BF16;
  if (encode_map_rows(&la.tm_do, b.dout, d, dq_dims[2], a.heads, tb, st[3], bwd_query_rows(d), bf16,
                      pr.key.merged != 0))
    return FA2_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(b.workspace);
  if (encode_dq_accum_map(&la.tm_dq, w, plan.slices, plan.rows_q, d)) return FA2_ERR_CUDA;
  BwdParams& p = la.p;
  p.f = pr.p;
  p.f.n_k = a.seqlen_k;   // packed: the longest sequence's key count the grid covers
  p.q = a.q;
  p.v = a.v;
  p.dout = b.dout;
  p.dq = b.dq;
  p.dk = b.dk;
  p.dv = b.dv;
  p.dq_accum = reinterpret_cast<float*>(w);
  p.delta = reinterpret_cast<float*>(w + plan.accum_bytes);
  p.q_bs = packed ? 0 : st[0][0];
  p.q_hs = st[0][1];
  p.q_rs = st[0][2];
  p.k_bs = packed ? 0 : st[1][0];
  p.k_hs = st[1][1];
  p.k_rs = st[1][2];
  p.v_bs = packed ? 0 : st[2][0];
  p.v_hs = st[2][1];
  p.v_rs = st[2][2];
  p.slices = plan.slices;
  p.num_k_tiles = plan.num_k_tiles;
  p.f.packed_units = (int)packed_grid_units(a, a.total_k, 128, plan.num_k_tiles);   // <= the plain grid
  p.scale = a.scale;
  la.bf16 = bf16;
  la.stream = stream;
  const int e = (d == 64) ? launch_bwd_d64(la) : (d == 128) ? launch_bwd_d128(la) : launch_bwd_d256(la);
  return e == 0 ? FA2_OK : FA2_ERR_CUDA;
}

}  // namespace
}  // namespace fa2

extern "C" size_t fa2_bwd_ex_workspace_bytes(const fa2_fwd_params* fwd) {
  if (!fwd) return 0;
  BwdPlan plan;
  if (bwd_plan(fold_batches(*fwd), plan)) return 0;
  return plan.accum_bytes + plan.delta_bytes;
}

extern "C" int fa2_bwd_ex(const fa2_bwd_params* params, void* stream) {
  if (!params) return FA2_ERR_INVALID_ARG;
  return backward(*params, static_cast<cudaStream_t>(stream));
}

extern "C" size_t fa2_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  const size_t rows = (size_t)B * H * (size_t)N;
  return align256(rows * (size_t)d * 4) + align256(rows * 4);
}

extern "C" int fa2_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                       void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N,
                       int d, float scale, int causal, int dtype, void* stream) {
  int rc = check_shape(B, H, N, d, scale, causal, dtype);
  if (rc) return rc;
  const void* ptrs[10] = {q, k, v, o, lse, dout, dq, dk, dv, workspace};
  for (const void* ptr : ptrs)
    if (!ptr) return FA2_ERR_INVALID_ARG;
  for (const void* ptr : ptrs)
    if (misaligned(ptr)) return FA2_ERR_MISALIGNED;
  fa2_bwd_params b;
  std::memset(&b, 0, sizeof(b));
  fa2_fwd_params& a = b.fwd;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = const_cast<void*>(o);
  a.lse = const_cast<float*>(lse);
  a.batch = B;
  a.heads = H;
  a.seqlen_q = N;
  a.seqlen_k = N;
  a.head_dim = d;
  a.dtype = dtype;
  a.scale = scale;
  a.window_left = -1;
  a.window_right = causal ? 0 : -1;
  const long long row = d, head = (long long)N * d, batch = (long long)H * N * d;
  int64_t* st[4] = {a.q_strides, a.k_strides, a.v_strides, a.o_strides};
  for (int64_t* s : st) {
    s[0] = batch;
    s[1] = head;
    s[2] = row;
  }
  a.lse_strides[0] = (long long)H * N;
  a.lse_strides[1] = N;
  b.dout = dout;
  b.dq = dq;
  b.dk = dk;
  b.dv = dv;
  b.workspace = workspace;
  b.workspace_bytes = workspace_bytes;
  return backward(b, static_cast<cudaStream_t>(stream));
}

extern "C" int fa2_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return FA2_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc) return rc;
  selftest_wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ds->status,
                                                                                (uint64_t)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

extern "C" int fa2_get_device_status(void* stream, uint32_t* detail) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA2_ERR_CUDA;
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc) return rc;
  uint32_t word = 0, zero = 0;
  if (cudaMemcpy(&word, ds->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return FA2_ERR_CUDA;
  if (word && cudaMemcpy(ds->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return FA2_ERR_CUDA;
  if (detail) *detail = word;
  if (word & kStatusTimeout) return FA2_ERR_DEVICE_TIMEOUT;
  if (word & kStatusBadSeqlens) return FA2_ERR_DEVICE_SEQLENS;
  return word ? FA2_ERR_DEVICE_TIMEOUT : FA2_OK;
}

extern "C" const char* fa2_status_string(int status) {
  switch (status) {
    case FA2_OK: return "ok";
    case FA2_ERR_INVALID_ARG: return "invalid argument (size, dtype, scale, null pointer or overlapping buffers)";
    case FA2_ERR_UNSUPPORTED: return "unsupported (head dim not 64/128/256, size limit, or not an sm_103 device)";
    case FA2_ERR_MISALIGNED: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case FA2_ERR_CUDA: return "CUDA runtime or driver call failed";
    case FA2_ERR_DEVICE_TIMEOUT: return "a kernel wait timed out; the tile was abandoned";
    case FA2_ERR_SCRATCH_LIMIT: return "problem exceeds the static device scratch of fa2_fwd_host_noalloc";
    case FA2_ERR_DEVICE_SEQLENS: return "packed-batch row offsets out of range; those sequences were not written";
    default: return "unknown status";
  }
}

extern "C" int fa2_version(void) { return 100; }
