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

struct KernelParams {
  void* o;            // [B,H,N,d] 16-bit output
  float* lse;         // [B,H,N] float32 output
  uint32_t* status;   // device status word (library-owned)
  int n;              // sequence length N
  int num_q_tiles;    // ceil(N / 128)
  int bh;             // B * H
  float scale_log2;   // scale * log2(e): scores go to the exp2 domain
};

struct LaunchArgs {
  CUtensorMap tm_q, tm_k, tm_v;
  KernelParams p;
  bool bf16;
  bool causal;
  cudaStream_t stream;
};

struct BwdParams {
  const float* lse;    // [B,H,N] forward logsumexp (natural log)
  const float* delta;  // [B,H,N] D_i = rowsum(dO_i o O_i), from the preprocess kernel
  float* dq_accum;     // [B,H,N,d] fp32, zeroed by the preprocess kernel
  void* dk;            // [B,H,N,d] 16-bit outputs
  void* dv;
  uint32_t* status;
  int n;
  int bh;
  int num_tiles;       // ceil(N / 128): key tiles = query tiles
  float scale;
  float scale_log2;
};

struct BwdLaunchArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // boxes of 64 columns x 128 rows
  CUtensorMap tm_dq;                    // fp32 dQ accumulator, boxes of 32 columns x 32 rows
  BwdParams p;
  const void* o;       // forward output, for D
  const void* dout;    // upstream gradient
  void* dq;            // 16-bit dQ output
  bool bf16;
  bool causal;
  cudaStream_t stream;
};

int launch_bwd_d64(const BwdLaunchArgs& a);
int launch_bwd_d128(const BwdLaunchArgs& a);

// Host-side tile geometry the launcher needs to build tensor maps: rows of Q
// per CTA tile and rows of K/V per streamed tile, per head dim.
struct TileGeometry {
  int q_rows;
  int kv_rows;
};

TileGeometry tile_geometry(int d);

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

}  // namespace fa2
