// fa2_internal.h -- declarations shared by the C-ABI translation unit and the
// per-head-dim kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa2 {

// Status bits a kernel ORs into the device status word when a bounded wait
// gives up: bit 0 = some wait timed out; bits 8..15 = wait site (role and
// barrier, see the kernel's WaitSite); the host maps any nonzero word to
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

// Host-side tile geometry the launcher needs to build tensor maps: rows of Q
// per CTA tile and rows of K/V per streamed tile, per head dim.
struct TileGeometry {
  int q_rows;
  int kv_rows;
};

TileGeometry tile_geometry(int d);

// Each launches the forward kernel for one head dim; returns a cudaError_t.
int launch_fwd_d64(const LaunchArgs& a);
int launch_fwd_d128(const LaunchArgs& a);
int launch_fwd_d256(const LaunchArgs& a);

}  // namespace fa2
