// FP8 E4M3 row-scaled GEMM entry point (ninfer PR #167: the row-scaled A8
// GEMM with linear / linear_add / linear_swiglu epilogues).
#include "gemm_launch.cuh"

using namespace spg;

namespace {

template <int EPI>
spg_status dispatch(const spg_route& r, const GemmMaps& m, const GemmParams& p, cudaStream_t s) {
  if constexpr (EPI != SPG_EPI_SWIGLU) {
    if (r.swap_ab) {
      // linear_add gives one ring stage to its residual blocks.
      constexpr bool kAdd = EPI == SPG_EPI_ADD;
      if (r.variant == 8) {
        if (r.block_n == 64)
          return launch_gemm_2sm_variant<EPI, 64, kAdd ? 9 : 10, false, false, kScaleRow, true,
                                         true>(m, p, r.grid, s);
        return launch_gemm_2sm_variant<EPI, 128, kAdd ? 7 : 8, false, false, kScaleRow, true,
                                       true>(m, p, r.grid, s);
      }
      if (r.block_n == 64)
        return launch_gemm_2sm_variant<EPI, 64, kAdd ? 9 : 10, false, false, kScaleRow, true>(
            m, p, r.grid, s);
      return launch_gemm_2sm_variant<EPI, 128, kAdd ? 7 : 8, false, false, kScaleRow, true>(
          m, p, r.grid, s);
    }
  }
  if (r.block_m == 256) {
    if (r.block_n == 192)
      return launch_gemm_2sm_variant<EPI, 192, 7, false, false, kScaleRow>(m, p, r.grid, s);
    if constexpr (EPI != SPG_EPI_SWIGLU) {
      if (r.block_n == 160)
        return launch_gemm_2sm_variant<EPI, 160, 7, false, false, kScaleRow>(m, p, r.grid, s);
    }
    if (r.block_n == 128)
      return launch_gemm_2sm_variant<EPI, 128, 8, false, false, kScaleRow>(m, p, r.grid, s);
    return launch_gemm_2sm_variant<EPI, 256, 6, false, false, kScaleRow>(m, p, r.grid, s);
  }
  if (r.block_n == 256)
    return launch_gemm_variant<kKindFp8, EPI, 256, 4, false, false, kScaleRow>(m, p, r.grid, s);
  return launch_gemm_variant<kKindFp8, EPI, 128, 6, false, false, kScaleRow>(m, p, r.grid, s);
}

}  // namespace

namespace {

spg_status rowscaled_impl(const uint8_t* A, const float* sa, const uint8_t* W, const float* sw,
                          const void* bias, const float* bias_scale, const void* residual, void* Y,
                          int64_t T, int64_t N, int64_t K, int epilogue, void* workspace,
                          int64_t workspace_bytes, spg_stream_t stream) {
  if (T < 0 || N < 0 || K < 0 || epilogue < 0 || epilogue > 2 || workspace_bytes < 0)
    return SPG_ERR_INVALID_ARG;
  if (T == 0 || N == 0) return SPG_OK;
  if (!A || !sa || !W || !sw || !Y || (epilogue == SPG_EPI_ADD && !residual))
    return SPG_ERR_INVALID_ARG;
  if (K == 0 || K % 16 != 0 || N % 8 != 0 || (epilogue == SPG_EPI_SWIGLU && N % 16 != 0) ||
      T > kMaxDim || N > kMaxDim || K > kMaxDim)
    return SPG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(A) || !aligned16(sa) || !aligned16(W) || !aligned16(sw) || !aligned16(Y) ||
      (epilogue == SPG_EPI_ADD && !aligned16(residual)) || !aligned16(workspace))
    return SPG_ERR_MISALIGNED;

  const spg_route r = route_for(SPG_KIND_FP8_ROWSCALED, T, N, K, epilogue, 1, false, workspace,
                                workspace_bytes);
  if (r.swap_ab) {
    // Swapped narrow-T tile: A operand = the weights (256 rows per pair
    // tile), B operand = the activations (block_n tokens); the epilogue
    // writes Y [T, N] transposed from the accumulator.
    GemmMaps maps;
    const uint32_t t_rows = static_cast<uint32_t>(r.block_n / 2);
    if (!make_tmap_3d(&maps.a, W, false, K, N, 1, K, K * N, 128, 128, 128) ||
        !make_tmap_3d(&maps.b, A, false, K, T, 1, K, K * T, 128, t_rows, 128) ||
        !make_tmap_3d(&maps.y, Y, true, N, T, 1, N * 2, N * 2 * T, 32, 32, 64))
      return SPG_ERR_CUDA;
    // The fourth map: the residual, as 32 x 32 blocks like the output.
    if (epilogue == SPG_EPI_ADD) {
      if (!make_tmap_3d(&maps.b_narrow, residual, true, N, T, 1, N * 2, N * 2 * T, 32, 32, 64))
        return SPG_ERR_CUDA;
    } else {
      maps.b_narrow = maps.b;
    }
    maps.r = maps.y;  // unused by the swapped tile
    GemmParams p;
    fill_common_params(p, r, N, T, K, K, N, 1);
    if (!p.err) return SPG_ERR_CUDA;
    if (const spg_status bs = set_bias(p, bias, bias_scale); bs != SPG_OK) return bs;
    const int pairs = num_sms() / 2;
    if (r.variant == 8)
      plan_pair_cluster_items(p, r, pairs);
    else
      plan_items(p, r, pairs, workspace);
    spg_route rr = r;
    rr.grid = 2 * (p.total_items < pairs ? p.total_items : pairs);
    p.row_scale = sw;
    p.col_scale = sa;
    p.residual = static_cast<const __nv_bfloat16*>(residual);
    if (epilogue == SPG_EPI_ADD) return dispatch<SPG_EPI_ADD>(rr, maps, p, stream);
    return dispatch<SPG_EPI_LINEAR>(rr, maps, p, stream);
  }
  const int b_rows = r.block_m == 256 ? r.block_n / 2 : r.block_n;  // B rows staged per CTA
  const int64_t n_out = epilogue == SPG_EPI_SWIGLU ? N / 2 : N;
  GemmMaps maps;
  if (!make_tmap_3d(&maps.a, A, false, K, T, 1, K, K * T, 128, 128, 128) ||
      !make_tmap_3d(&maps.b, W, false, K, N, 1, K, K * N, 128, b_rows, 128) ||
      !make_tmap_3d(&maps.y, Y, true, n_out, T, 1, n_out * 2, n_out * 2 * T, 32, 32, 64))
    return SPG_ERR_CUDA;
  maps.r = maps.y;
  if (r.block_m == 256 && epilogue == SPG_EPI_ADD &&
      !make_tmap_3d(&maps.r, residual, true, N, T, 1, N * 2, N * 2 * T, 32, 32, 64))
    return SPG_ERR_CUDA;
  GemmParams p;
  fill_common_params(p, r, T, N, K, K, n_out, 1);
  if (!p.err) return SPG_ERR_CUDA;
  if (const spg_status bs = set_bias(p, bias, bias_scale); bs != SPG_OK) return bs;
  spg_route rr = r;
  if (r.block_m == 256) {
    const int pairs = num_sms() / 2;
    plan_items(p, r, pairs, workspace);
    rr.grid = 2 * (p.total_items < pairs ? p.total_items : pairs);
    const uint32_t narrow_rows = static_cast<uint32_t>(r.block_n / p.split_ways / 2);
    if (!make_tmap_3d(&maps.b_narrow, W, false, K, N, 1, K, K * N, 128, narrow_rows, 128))
      return SPG_ERR_CUDA;
  }
  p.row_scale = sa;
  p.col_scale = sw;
  p.residual = static_cast<const __nv_bfloat16*>(residual);
  switch (epilogue) {
    case SPG_EPI_LINEAR: return dispatch<SPG_EPI_LINEAR>(rr, maps, p, stream);
    case SPG_EPI_ADD: return dispatch<SPG_EPI_ADD>(rr, maps, p, stream);
    default: return dispatch<SPG_EPI_SWIGLU>(rr, maps, p, stream);
  }
}

}  // namespace

extern "C" spg_status fp8_rowscaled_gemm(const uint8_t* A, const float* sa, const uint8_t* W,
                                         const float* sw, const void* residual, void* Y,
                                         int64_t T, int64_t N, int64_t K, int epilogue,
                                         spg_stream_t stream) {
  return rowscaled_impl(A, sa, W, sw, nullptr, nullptr, residual, Y, T, N, K, epilogue, nullptr, 0,
                        stream);
}

extern "C" spg_status fp8_rowscaled_gemm_bias(const uint8_t* A, const float* sa, const uint8_t* W,
                                              const float* sw, const void* bias,
                                              const float* bias_scale, const void* residual,
                                              void* Y, int64_t T, int64_t N, int64_t K,
                                              int epilogue, spg_stream_t stream) {
  return rowscaled_impl(A, sa, W, sw, bias, bias_scale, residual, Y, T, N, K, epilogue, nullptr, 0,
                        stream);
}

extern "C" spg_status fp8_rowscaled_gemm_ws(const uint8_t* A, const float* sa, const uint8_t* W,
                                            const float* sw, const void* bias,
                                            const float* bias_scale, const void* residual, void* Y,
                                            int64_t T, int64_t N, int64_t K, int epilogue,
                                            void* workspace, int64_t workspace_bytes,
                                            spg_stream_t stream) {
  return rowscaled_impl(A, sa, W, sw, bias, bias_scale, residual, Y, T, N, K, epilogue, workspace,
                        workspace_bytes, stream);
}
