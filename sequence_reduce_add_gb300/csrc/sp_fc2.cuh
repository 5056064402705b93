// sp_fc2.cuh — FlashComm2 token reorganisation on one GPU (vllm-ascend SP/FlashComm notes
// §4.2-4.4): all G = global_tp ranks' [N][H/G] feature slices live in one buffer x [G][N][F]
// (F = H/G); the output y [G][N/D][D*F] (D = odp_size = G/P, P = otp_size) is what every rank
// holds after the local reorder by the reorganised batch ids, the ODP-group all_to_all and the
// feature concat.
//
// Closed form of that map: output rank r = g*D + j, output row i = k*S + tl (S = N/G tokens
// per segment, k < P, tl < S), feature block m < D  <-  source rank g*D + m, source token
// (j + k*D)*S + tl, all F features. Each such (r, i, m) piece is F contiguous elements on both
// sides; pieces are numbered in output order, so the writes stream sequentially.
#pragma once

#include "sp_device.cuh"

namespace spk {

struct Fc2Params {
  const unsigned char* x;
  unsigned char* y;
  int64_t N;           // tokens
  int64_t pieces;      // G * N: pieces of F elements
  int64_t S;           // tokens per segment, N / G
  int D;               // odp_size
  int P;               // otp_size
  int piece_vecs;      // F * elem_bytes / 16
};

constexpr int kFc2Threads = 256;

__global__ void __launch_bounds__(kFc2Threads) k_fc2_reorganize(const Fc2Params p) {
  pdl_launch_dependents();
  pdl_wait_prerequisites();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kFc2Threads / 32);
  const int64_t per_rank = p.S * p.P * p.D;  // pieces per output rank
  for (int64_t piece = static_cast<int64_t>(blockIdx.x) * (kFc2Threads / 32) + (threadIdx.x >> 5);
       piece < p.pieces; piece += warps) {
    const int64_t r = piece / per_rank;
    const int64_t rem = piece - r * per_rank;
    const int64_t i = rem / p.D;
    const int m = static_cast<int>(rem - i * p.D);
    const int64_t g = r / p.D, j = r - g * p.D;
    const int64_t k = i / p.S, tl = i - k * p.S;
    const int64_t src_rank = g * p.D + m;
    const int64_t src_token = (j + k * p.D) * p.S + tl;
    const uint4* src = reinterpret_cast<const uint4*>(p.x) + (src_rank * p.N + src_token) * p.piece_vecs;
    uint4* dst = reinterpret_cast<uint4*>(p.y) + piece * p.piece_vecs;
    // 128 vectors (2 KB) per pass: every lane issues all of its (up to four) loads before its
    // first store, so each warp keeps up to 2 KB in flight.
    for (int base = 0; base < p.piece_vecs; base += 128) {
      uint4 buf[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = base + lane + 32 * u;
        if (v < p.piece_vecs) buf[u] = ldg_stream(src + v);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = base + lane + 32 * u;
        if (v < p.piece_vecs) stg_stream(dst + v, buf[u]);
      }
    }
  }
}

}  // namespace spk
