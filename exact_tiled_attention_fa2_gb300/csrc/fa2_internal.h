// fa2_internal.h -- declarations shared by the C-ABI translation unit and the
// per-head-dim kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace fa2 {

// Status bits a kernel ORs into the device status word when a bounded wait
// gives up: bit 0 = some wait timed out; bit 8 + s for each wait site s that
// gave up (see WaitSite); the host maps any nonzero word to
// FA2_ERR_DEVICE_TIMEOUT.
constexpr uint32_t kStatusTimeout = 1u;

// Forward-pass arguments the kernels read.  Element (b, h, i) of O lives at
// o + b*o_bs + h*o_hs + (row0_q(b) + i)*o_rs elements, of LSE at
// lse + b*l_bs + h*l_hs + row0_q(b) + i, where row0_q(b) is cu_q[b] for packed
// variable-length batches and 0 otherwise (keys: cu_k[b] and 0).
struct KernelParams {
  void* o;            // 16-bit output
  float* lse;         // float32 output
  uint32_t* status;   // device status word (library-owned)
  const int* cu_q;    // [B+1] query row offsets of packed sequences, or null
  const int* cu_k;    // [B+1] key row offsets, or null (set iff cu_q is)
  long long o_bs, o_hs, o_rs;  // O strides in elements (head-dim stride 1)
  long long l_bs, l_hs;        // LSE strides in elements (row stride 1)
  int n_q;            // query rows per sequence (packed: the maximum)
  int n_k;            // keys per sequence (packed: the maximum)
  int total_q;        // packed: rows of q/o/lse (bound for cu_q); else n_q
  int total_k;        // packed: rows of k/v (bound for cu_k); else n_k
  int heads;          // H
  int merged_bh;      // 1: the tensor maps are 3-D (d, rows, B*H), coordinate b*H + h; 0: 4-D
  int tma_o;          // 1: O is staged in shared memory and written by TMA stores (unpacked batches)
  int bh;             // B * H
  int units;          // work units per (b, h): query tiles (split-key mode: tiles x chunks)
  int window_left;    // key j visible to query i iff i+off-wl <= j <= i+off+wr
  int window_right;   //   (off = N_k - N_q; -1 = unbounded on that side),
  int prefix;         //   or j < prefix (keys every query sees)
  float scale_log2;   // scale * log2(e), signed: scores go to the exp2 domain
  // The tiled forward kernel's form of the scale: it scales raw scores by
  // scale_log2_mag = max(|scale * log2(e)|, FLT_MIN) and, for a negative
  // scale, negates the S product (qk_negate: the negate-A bit of its
  // instruction descriptor, else 0).  FLT_MIN in place of a zero scale rounds
  // every scaled score to zero against the row maximum (P = 1 on every
  // visible key, exactly as with scale 0) and keeps a hidden key's -inf from
  // forming -inf * 0.
  float scale_log2_mag;
  uint32_t qk_negate;
  // Split-key mode of the double-buffered kernel (decoding): a unit is a
  // (query tile, key chunk) pair, and each row's partial (m, l, O~) goes to
  // ws_ml / ws_o in the decode merge kernel's layout instead of O and LSE.
  int splits;         // key chunks per (b, h); 0 or 1: whole rows
  int split_chunk;    // keys per chunk, a multiple of the key tile
  int split_base;     // first key of chunk 0 (a multiple of the key tile)
  float* ws_o;        // [B*H][n_q][splits][d] partial O~
  float* ws_ml;       // [B*H][n_q][splits][2] partial (m, l), exp2 domain
  int packed_units;   // packed batches of at most kPackedScanSeqs sequences: units per head over
                      // all sequences (the grid is heads x packed_units); 0: bh x units
};

// Bit of the status word a forward kernel sets when a packed batch's row
// offsets are out of range; that sequence is left unwritten.
constexpr uint32_t kStatusBadSeqlens = 2u;

// Packed batches of up to this many sequences launch only the tiles that
// exist (each CTA's threads read one sequence's offsets each).
constexpr int kPackedScanSeqs = 192;

struct LaunchArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // (d, rows, B*H) or (d, rows, H, B) maps, boxes of 64 columns
  CUtensorMap tm_o;              // the same view of o, boxes of 64 columns x 32 rows (one warp's rows)
  KernelParams p;
  bool bf16;
  bool band;  // window_left >= 0 or prefix > 0: a row's first visible key depends on the row
  cudaStream_t stream;
};

// Backward-pass arguments the kernels read.  Sequence offsets, strides and
// sizes follow KernelParams (`f`): dout has o's layout, dq q's, dk k's and dv
// v's.  Per (tensor batch, head) slice hb = b*H + h the workspace holds D
// [hb][rows_q] and the fp32 dQ accumulator [hb][rows_q][d], rows_q = f.total_q.
struct BwdParams {
  KernelParams f;       // o and lse are the forward's outputs here (read)
  const void* q;        // read by the preprocess (nothing) and the kernels via maps
  const void* v;        // read directly by the d = 256 kernel (V_j into tensor memory)
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  const float* delta;   // D_i = rowsum(dO_i o O_i), from the preprocess kernel
  float* dq_accum;      // zeroed by the preprocess kernel
  long long q_bs, q_hs, q_rs;   // q (= dq) strides
  long long k_bs, k_hs, k_rs;   // k (= dk) strides
  long long v_bs, v_hs, v_rs;   // v (= dv) strides
  long long slices;     // (tensor batch) x heads: 1 x H for packed batches, B x H otherwise
  int num_k_tiles;      // key tiles per (b, h), from the longest key sequence
  float scale;
};

struct BwdLaunchArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // boxes of 64 columns x 128 rows
  CUtensorMap tm_dq;                    // fp32 dQ accumulator, boxes of 32 columns x 32 rows
  BwdParams p;
  bool bf16;
  cudaStream_t stream;
};

int launch_bwd_d64(const BwdLaunchArgs& a);
int launch_bwd_d128(const BwdLaunchArgs& a);
int launch_bwd_d256(const BwdLaunchArgs& a);

// Host-side tile geometry the launcher needs to build tensor maps and size
// the grid: rows of Q per tile, rows of K/V per streamed tile and query rows
// per CTA, per head dim.
struct TileGeometry {
  int q_rows;
  int kv_rows;
  int cta_rows;
};

TileGeometry tile_geometry(int d);

// Key rows per pipeline stage of the decode kernel (the box height of its
// K/V tensor maps).
constexpr int decode_block_rows(int d) { return d == 256 ? 32 : 64; }

// One-time per-device set-up of a kernel instantiation (attributes, checks):
// `setup` runs until it succeeds once on a device; devices >= 64 run it on
// every call.
template <class F>
inline int once_per_device(std::atomic<unsigned long long>& done, F&& setup) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return (int)cudaErrorNoDevice;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return 0;
  const int e = setup();
  if (e == 0 && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Each launches the forward kernel for one head dim; returns a cudaError_t.
int launch_fwd_d64(const LaunchArgs& a);
int launch_fwd_d128(const LaunchArgs& a);
int launch_fwd_d256(const LaunchArgs& a);

struct DecodeLaunchArgs;
int launch_decode_d64(const DecodeLaunchArgs& a);
int launch_decode_d256(const DecodeLaunchArgs& a);
// Decoding on the tensor cores (3 or more query rows, d = 64 / 128, unpacked):
// the double-buffered forward kernel in split-key mode, then the decode merge
// kernel.  `a.p` carries the split fields; maps: q boxes of 128 rows, k and v
// boxes of 64 rows.
int launch_decode_tc_d64(const LaunchArgs& a);
int launch_decode_tc_d128(const LaunchArgs& a);

}  // namespace fa2
