// NVFP4 block-scaled GEMM entry point (ninfer PR #160: E2M1 codes with an
// E4M3 scale per 16 elements, scale tiles loaded whole, linear_add and the
// fused SwiGLU route).
#include "gemm_launch.cuh"
#include "gemv_nvfp4.cuh"

using namespace spg;

namespace {

template <int EPI>
spg_status launch(const spg_route& r, const GemmMaps& m, const GemmParams& p, cudaStream_t s) {
  if (r.block_m == 256 && r.variant == 5) {
    if (p.bias_kind) return launch_nvfp4_mc_variant<EPI, 3, true>(m, p, r.grid, s);
    return launch_nvfp4_mc_variant<EPI, 3, false>(m, p, r.grid, s);
  }
  if (r.block_m == 256 && r.variant == 3) {
    if (p.bias_kind) return launch_nvfp4_2sm_st_variant<EPI, 5, true>(m, p, r.grid, s);
    return launch_nvfp4_2sm_st_variant<EPI, 5, false>(m, p, r.grid, s);
  }
  if (r.block_m == 256) {
    if (p.bias_kind) return launch_nvfp4_2sm_variant<EPI, 5, true>(m, p, r.grid, s);
    return launch_nvfp4_2sm_variant<EPI, 5, false>(m, p, r.grid, s);
  }
  if (r.variant == 7) {
    if (r.block_n == 256)
      return launch_gemm_csplit_variant<kKindNvfp4, EPI, 256, 3, false, false, kScaleScalar>(m, p, s);
    return launch_gemm_csplit_variant<kKindNvfp4, EPI, 128, 5, false, false, kScaleScalar>(m, p, s);
  }
  return launch_gemm_variant<kKindNvfp4, EPI, 128, 5, false, false, kScaleScalar>(m, p, r.grid, s);
}

}  // namespace

namespace {

spg_status nvfp4_impl(const uint8_t* A, const uint8_t* sfA, const float* gA, const uint8_t* W,
                      const uint8_t* sfW, const float* gW, const void* bias,
                      const float* bias_scale, const void* residual, void* Y, int64_t T,
                      int64_t N, int64_t K, int epilogue, void* workspace,
                      int64_t workspace_bytes, spg_stream_t stream) {
  if (T < 0 || N < 0 || K < 0 || epilogue < 0 || epilogue > 2 || workspace_bytes < 0)
    return SPG_ERR_INVALID_ARG;
  if (T == 0 || N == 0) return SPG_OK;
  if (!A || !sfA || !gA || !W || !sfW || !gW || !Y || (epilogue == SPG_EPI_ADD && !residual))
    return SPG_ERR_INVALID_ARG;
  if (K == 0 || K % 256 != 0 || N % 8 != 0 || (epilogue == SPG_EPI_SWIGLU && N % 16 != 0) ||
      T > kMaxDim || N > kMaxDim || K > kMaxDim)
    return SPG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(A) || !aligned16(sfA) || !aligned16(gA) || !aligned16(W) || !aligned16(sfW) ||
      !aligned16(gW) || !aligned16(Y) || (epilogue == SPG_EPI_ADD && !aligned16(residual)) ||
      !aligned16(workspace))
    return SPG_ERR_MISALIGNED;

  const spg_route r =
      route_for(SPG_KIND_NVFP4, T, N, K, epilogue, 1, false, workspace, workspace_bytes);
  if (r.variant == 4) {
    // Decode-sized T: the CUDA-core GEMV (no tensor maps, no workspace).
    GemvParams g;
    g.A = A;
    g.sfA = sfA;
    g.gA = gA;
    g.X = nullptr;
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
    return launch_gemv_epilogue(g, epilogue, stream);
  }
  const int64_t kh = K / 2;
  const int64_t n_out = epilogue == SPG_EPI_SWIGLU ? N / 2 : N;
  GemmMaps maps;
  // B box: the rows one CTA stages per stage (a pair tile's CTA stages half
  // of its 256 rows; a one-CTA tile all of block_n).
  const uint32_t b_rows = r.block_m == 256 ? 128u : static_cast<uint32_t>(r.block_n);
  if (!make_tmap_3d(&maps.a, A, false, kh, T, 1, kh, kh * T, 128, 128, 128) ||
      !make_tmap_3d(&maps.b, W, false, kh, N, 1, kh, kh * N, 128, b_rows, 128) ||
      !make_tmap_3d(&maps.y, Y, true, n_out, T, 1, n_out * 2, n_out * 2 * T, 32, 32, 64))
    return SPG_ERR_CUDA;
  if (r.block_m == 256) {
    // Scale buffers as 2-D [tiles, 128 x uint32] views: one row per 512-byte tile.
    const uint64_t tpr = static_cast<uint64_t>(K / 64);
    const uint64_t tiles_a = static_cast<uint64_t>((T + 127) / 128) * tpr;
    const uint64_t tiles_b = static_cast<uint64_t>((N + 127) / 128) * tpr;
    if (!make_tmap_2d_u32(&maps.sfa, sfA, 128, tiles_a, 512, 128, 4) ||
        !make_tmap_2d_u32(&maps.sfb, sfW, 128, tiles_b, 512, 128, 4))
      return SPG_ERR_CUDA;
    if (epilogue == SPG_EPI_ADD) {
      if (!make_tmap_3d(&maps.r, residual, true, N, T, 1, N * 2, N * 2 * T, 32, 32, 64))
        return SPG_ERR_CUDA;
    } else {
      maps.r = maps.y;
    }
  }
  GemmParams p;
  fill_common_params(p, r, T, N, kh, K, n_out, 1);
  if (!p.err) return SPG_ERR_CUDA;
  if (const spg_status bs = set_bias(p, bias, bias_scale); bs != SPG_OK) return bs;
  p.scalar_a = gA;
  p.scalar_b = gW;
  p.residual = static_cast<const __nv_bfloat16*>(residual);
  p.sfa = sfA;
  p.sfb = sfW;
  p.sf_tiles_per_row_block = static_cast<int>(K / 64);
  spg_route rr = r;
  if (r.block_m == 256) {
    const int pairs = num_sms() / 2;
    plan_items(p, r, pairs, workspace);
    rr.grid = 2 * (p.total_items < pairs ? p.total_items : pairs);
  } else if (r.variant == 7) {
    const int ring = r.stages * (128 * 128 + r.block_n * 128 + 2048 + (r.block_n / 128) * 2048);
    plan_cluster_items(p, r, ring, epilogue == SPG_EPI_SWIGLU ? 64 : 32);
  }
  switch (epilogue) {
    case SPG_EPI_LINEAR: return launch<SPG_EPI_LINEAR>(rr, maps, p, stream);
    case SPG_EPI_ADD: return launch<SPG_EPI_ADD>(rr, maps, p, stream);
    default: return launch<SPG_EPI_SWIGLU>(rr, maps, p, stream);
  }
}

}  // namespace

extern "C" spg_status nvfp4_gemm(const uint8_t* A, const uint8_t* sfA, const float* gA,
                                 const uint8_t* W, const uint8_t* sfW, const float* gW,
                                 const void* residual, void* Y, int64_t T, int64_t N, int64_t K,
                                 int epilogue, spg_stream_t stream) {
  return nvfp4_impl(A, sfA, gA, W, sfW, gW, nullptr, nullptr, residual, Y, T, N, K, epilogue,
                    nullptr, 0, stream);
}

extern "C" spg_status nvfp4_gemm_bias(const uint8_t* A, const uint8_t* sfA, const float* gA,
                                      const uint8_t* W, const uint8_t* sfW, const float* gW,
                                      const void* bias, const float* bias_scale,
                                      const void* residual, void* Y, int64_t T, int64_t N,
                                      int64_t K, int epilogue, spg_stream_t stream) {
  return nvfp4_impl(A, sfA, gA, W, sfW, gW, bias, bias_scale, residual, Y, T, N, K, epilogue,
                    nullptr, 0, stream);
}

extern "C" spg_status nvfp4_gemm_ws(const uint8_t* A, const uint8_t* sfA, const float* gA,
                                    const uint8_t* W, const uint8_t* sfW, const float* gW,
                                    const void* bias, const float* bias_scale,
                                    const void* residual, void* Y, int64_t T, int64_t N, int64_t K,
                                    int epilogue, void* workspace, int64_t workspace_bytes,
                                    spg_stream_t stream) {
  return nvfp4_impl(A, sfA, gA, W, sfW, gW, bias, bias_scale, residual, Y, T, N, K, epilogue,
                    workspace, workspace_bytes, stream);
}
