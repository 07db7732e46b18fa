// Activation operators: bf16 activations in, quantized inside the call,
// then the GEMM with its fused epilogue -- the "operator" the pages time
// (ninfer PR #160 "The NVFP4 TMA route reads activation scales as one
// tile": the operator table counts the bf16 activation read; ninfer PR #167
// "The fp8 A8 GEMM stages its operands through TMA": the A8 call sites
// quantize their activations per row at run time).
//
// The quantizer and the GEMM run back to back on the caller's stream, the
// codes and scales passing through the caller's workspace (NVFP4 at decode
// widths: the one-CTA global-scale-and-encode kernel, then the GEMV).  The
// library also has a single-kernel form for NVFP4 decode widths -- each CTA
// cluster of the GEMV quantizes the activations itself, in the order and
// precision of the block quantizer, into the shared planes it multiplies
// from -- pinned with SPG_FORCE_VARIANT=gemv_fused (measured slower than the
// two kernels; see nvfp4_fused_route).
#include <cuda_bf16.h>

#include "common.h"
#include "gemv_nvfp4.cuh"
#include "host.h"

using namespace spg;

namespace {

constexpr int64_t kAlign = 256;

int64_t round_up(int64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Workspace layout of an operator call: the activation codes and scales
// first, the GEMM's own K-split workspace after them.
struct ActLayout {
  int64_t codes = 0, scales = 0, scratch = 0, gemm = 0;  // byte offsets
  int64_t required = 0;  // bytes the activation part needs
  int64_t total = 0;     // with the GEMM's workspace
  bool fused = false;    // NVFP4 decode: one GEMV kernel, no workspace
};

// The fused decode kernel (the GEMV in its operator form) runs when
// SPG_FORCE_VARIANT=gemv_fused pins it.  It measured faster than the
// four-launch quantizer followed by the GEMV (SwiGLU N = 34816, T = 1 / 2:
// 47.6 / 51.7 against 52-56 us; linear_add N = 5120, K = 6144, T = 1: 21.0
// against 25.1), but not than the one-CTA quantizer (spg_quantize_nvfp4_act)
// followed by the plain route, which the operator now uses (45.5 / 49.6
// against 41.4 / 45.5; 20.9 against 18.9; GB300, graph-replayed, L2
// flushed): the cluster's quantization plus its two cluster barriers cost
// more than a one-CTA kernel whose latency overlaps the GEMV's start.
bool nvfp4_fused_route(int64_t T, int64_t N, int64_t K, int epilogue) {
  (void)N;
  if (T < 1 || T > 4 || epilogue < 0 || epilogue > 2) return false;
  if (T * (K / 32) * 34 > 200 * 1024) return false;  // the GEMV's shared memory
  return forced_variant_is("gemv_fused");
}

ActLayout act_layout(int kind, int64_t T, int64_t N, int64_t K, int epilogue) {
  ActLayout l;
  if (kind == SPG_KIND_NVFP4 && nvfp4_fused_route(T, N, K, epilogue)) {
    l.fused = true;
    return l;
  }
  int64_t off = 0;
  if (kind == SPG_KIND_FP8_ROWSCALED) {
    l.codes = off;
    off += round_up(T * K);
    l.scales = off;
    off += round_up(4 * T);
  } else {
    l.scratch = off;  // amax scratch at +0, global scale at +16
    off += kAlign;
    l.codes = off;
    off += round_up(T * K / 2);
    l.scales = off;
    off += round_up(static_cast<int64_t>(spg_nvfp4_sf_bytes(T, K)));
  }
  l.required = off;
  l.gemm = off;
  l.total = off + spg_gemm_workspace_bytes(kind, T, N, K, epilogue, 1);
  return l;
}

bool shape_ok(int64_t T, int64_t N, int64_t K) {
  return T >= 0 && N >= 0 && K >= 0 && T <= 0x7FFFFFFF && N <= 0x7FFFFFFF && K <= 0x7FFFFFFF;
}

}  // namespace

extern "C" int64_t spg_act_workspace_bytes(int kind, int64_t T, int64_t N, int64_t K,
                                           int epilogue) {
  if ((kind != SPG_KIND_FP8_ROWSCALED && kind != SPG_KIND_NVFP4) || T <= 0 || N <= 0 || K <= 0 ||
      epilogue < 0 || epilogue > 2 || !shape_ok(T, N, K))
    return 0;
  if (kind == SPG_KIND_NVFP4 && K % 64 != 0) return 0;
  return act_layout(kind, T, N, K, epilogue).total;
}

extern "C" spg_status fp8_rowscaled_linear_bf16(const void* X, const uint8_t* W, const float* sw,
                                                const void* bias, const float* bias_scale,
                                                const void* residual, void* Y, int64_t T,
                                                int64_t N, int64_t K, int epilogue,
                                                void* workspace, int64_t workspace_bytes,
                                                spg_stream_t stream) {
  if (!shape_ok(T, N, K) || epilogue < 0 || epilogue > 2 || workspace_bytes < 0)
    return SPG_ERR_INVALID_ARG;
  if (T == 0 || N == 0) return SPG_OK;
  if (!X || !workspace) return SPG_ERR_INVALID_ARG;
  if (K == 0 || K % 16 != 0) return SPG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(X) || !aligned16(workspace)) return SPG_ERR_MISALIGNED;
  const ActLayout l = act_layout(SPG_KIND_FP8_ROWSCALED, T, N, K, epilogue);
  if (workspace_bytes < l.required) return SPG_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* A = ws + l.codes;
  float* sa = reinterpret_cast<float*>(ws + l.scales);
  const spg_status q = spg_quantize_fp8_rows(X, T, K, A, sa, stream);
  if (q != SPG_OK) return q;
  return fp8_rowscaled_gemm_ws(A, sa, W, sw, bias, bias_scale, residual, Y, T, N, K, epilogue,
                               ws + l.gemm, workspace_bytes - l.gemm, stream);
}

extern "C" spg_status nvfp4_linear_bf16(const void* X, const uint8_t* W, const uint8_t* sfW,
                                        const float* gW, const void* bias,
                                        const float* bias_scale, const void* residual, void* Y,
                                        int64_t T, int64_t N, int64_t K, int epilogue,
                                        void* workspace, int64_t workspace_bytes,
                                        spg_stream_t stream) {
  if (!shape_ok(T, N, K) || epilogue < 0 || epilogue > 2 || workspace_bytes < 0)
    return SPG_ERR_INVALID_ARG;
  if (T == 0 || N == 0) return SPG_OK;
  if (!X) return SPG_ERR_INVALID_ARG;
  if (K == 0 || K % 256 != 0 || N % 8 != 0 || (epilogue == SPG_EPI_SWIGLU && N % 16 != 0))
    return SPG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(X) || !aligned16(workspace)) return SPG_ERR_MISALIGNED;
  const ActLayout l = act_layout(SPG_KIND_NVFP4, T, N, K, epilogue);
  if (l.fused) {
    if (!W || !sfW || !gW || !Y || (epilogue == SPG_EPI_ADD && !residual))
      return SPG_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(sfW) || !aligned16(gW) || !aligned16(Y) ||
        (epilogue == SPG_EPI_ADD && !aligned16(residual)))
      return SPG_ERR_MISALIGNED;
    GemvParams g;
    g.A = nullptr;
    g.sfA = nullptr;
    g.gA = nullptr;
    g.X = static_cast<const __nv_bfloat16*>(X);
    g.W = W;
    g.sfW = sfW;
    g.gW = gW;
    g.bias = bias;
    g.bias_scale = bias_scale;
    g.bias_kind = 0;
    if (bias) {
      if (!aligned16(bias) || (bias_scale && !aligned16(bias_scale))) return SPG_ERR_MISALIGNED;
      g.bias_kind = bias_scale ? 2 : 1;
    } else if (bias_scale) {
      return SPG_ERR_INVALID_ARG;
    }
    g.residual = static_cast<const __nv_bfloat16*>(residual);
    g.Y = static_cast<__nv_bfloat16*>(Y);
    g.T = static_cast<int>(T);
    g.N = static_cast<int>(N);
    g.K = static_cast<int>(K);
    g.n_out = static_cast<int>(epilogue == SPG_EPI_SWIGLU ? N / 2 : N);
    return launch_gemv_epilogue(g, epilogue, static_cast<cudaStream_t>(stream));
  }
  if (!workspace || workspace_bytes < l.required) return SPG_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* amax = reinterpret_cast<float*>(ws + l.scratch);
  float* gA = reinterpret_cast<float*>(ws + l.scratch + 16);
  uint8_t* A = ws + l.codes;
  uint8_t* sfA = ws + l.scales;
  const spg_status s = spg_quantize_nvfp4_act(X, T, K, gA, amax, A, sfA, stream);
  if (s != SPG_OK) return s;
  return nvfp4_gemm_ws(A, sfA, gA, W, sfW, gW, bias, bias_scale, residual, Y, T, N, K, epilogue,
                       ws + l.gemm, workspace_bytes - l.gemm, stream);
}
