// Per-tensor-scaled FP8 GEMM entry point, NT / NN / TN / TT, batched
// (AstrAI commit log of csrc/kernels/fp8/gemm.cuh: layout tags instead of
// copies, batch strides with stride 0 broadcasting, bf16 output).
// Non-K-major operands are read as MN-major shared-memory tiles, which the
// tensor core consumes directly (no transpose pass).
#include "gemm_launch.cuh"

using namespace spg;

namespace {

template <bool A_MN, bool B_MN>
spg_status dispatch(const spg_route& r, const GemmMaps& m, const GemmParams& p, cudaStream_t s) {
  if (r.block_m == 256) {
    if constexpr (!B_MN) {
      if (r.block_n == 192)
        return launch_gemm_2sm_variant<SPG_EPI_LINEAR, 192, 7, A_MN, B_MN, kScaleScalar>(m, p, r.grid, s);
      if (r.block_n == 160)
        return launch_gemm_2sm_variant<SPG_EPI_LINEAR, 160, 7, A_MN, B_MN, kScaleScalar>(m, p, r.grid, s);
      if (r.block_n == 128)
        return launch_gemm_2sm_variant<SPG_EPI_LINEAR, 128, 8, A_MN, B_MN, kScaleScalar>(m, p, r.grid, s);
    }
    return launch_gemm_2sm_variant<SPG_EPI_LINEAR, 256, 6, A_MN, B_MN, kScaleScalar>(m, p, r.grid, s);
  }
  if (r.block_n == 256)
    return launch_gemm_variant<kKindFp8, SPG_EPI_LINEAR, 256, 4, A_MN, B_MN, kScaleScalar>(m, p, r.grid, s);
  return launch_gemm_variant<kKindFp8, SPG_EPI_LINEAR, 128, 6, A_MN, B_MN, kScaleScalar>(m, p, r.grid, s);
}

}  // namespace

namespace {

spg_status tensor_impl(char layout_a, char layout_b, int64_t batch, const uint8_t* A,
                       int64_t strideA, const float* sA, const uint8_t* B, int64_t strideB,
                       const float* sB, const void* bias, const float* bias_scale, void* C,
                       int64_t strideC, int64_t M, int64_t N, int64_t K, void* workspace,
                       int64_t workspace_bytes, spg_stream_t stream) {
  if ((layout_a != 'N' && layout_a != 'T') || (layout_b != 'N' && layout_b != 'T'))
    return SPG_ERR_INVALID_ARG;
  if (batch < 0 || M < 0 || N < 0 || K < 0 || strideA < 0 || strideB < 0 || strideC < 0 ||
      workspace_bytes < 0)
    return SPG_ERR_INVALID_ARG;
  if (batch == 0 || M == 0 || N == 0) return SPG_OK;
  if (!A || !B || !C || !sA || !sB) return SPG_ERR_INVALID_ARG;
  const bool a_mn = layout_a == 'T';
  const bool b_mn = layout_b == 'N';
  if (K == 0 || K % 16 != 0 || N % 8 != 0 || (a_mn && M % 16 != 0) || (b_mn && N % 16 != 0) ||
      M > kMaxDim || N > kMaxDim || K > kMaxDim || batch > 65535)
    return SPG_ERR_UNSUPPORTED_SHAPE;
  if (batch > 1) {
    if (strideA % 16 != 0 || strideB % 16 != 0 || strideC % 8 != 0 || strideC < M * N ||
        (strideA != 0 && strideA < M * K) || (strideB != 0 && strideB < N * K))
      return SPG_ERR_UNSUPPORTED_SHAPE;
  }
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || !aligned16(sA) || !aligned16(sB) ||
      !aligned16(workspace))
    return SPG_ERR_MISALIGNED;

  // The swapped narrow-M tile reads both operands K-major ("NT" only).
  const spg_route r = route_for(SPG_KIND_FP8_TENSOR, M, N, K, SPG_EPI_LINEAR, batch, b_mn,
                                workspace, workspace_bytes, !a_mn);
  if (r.swap_ab) {
    // Swapped tile (M <= 128, one matrix): the MMA's 256-row side takes B's
    // rows (the output columns), its N side M rows of A; the epilogue writes
    // C [M, N] transposed from the accumulator, scaled by sA * sB.
    GemmMaps maps;
    const uint32_t t_rows = static_cast<uint32_t>(r.block_n / 2);
    if (!make_tmap_3d(&maps.a, B, false, K, N, 1, K, K * N, 128, 128, 128) ||
        !make_tmap_3d(&maps.b, A, false, K, M, 1, K, K * M, 128, t_rows, 128) ||
        !make_tmap_3d(&maps.y, C, true, N, M, 1, N * 2, N * 2 * M, 32, 32, 64))
      return SPG_ERR_CUDA;
    maps.b_narrow = maps.b;  // the swapped tile never splits along N
    maps.r = maps.y;         // no residual
    GemmParams p;
    fill_common_params(p, r, N, M, K, K, N, 1);
    if (!p.err) return SPG_ERR_CUDA;
    if (const spg_status bs = set_bias(p, bias, bias_scale); bs != SPG_OK) return bs;
    const int pairs = num_sms() / 2;
    if (r.variant == 8)
      plan_pair_cluster_items(p, r, pairs);
    else
      plan_items(p, r, pairs, workspace);
    spg_route rr = r;
    rr.grid = 2 * (p.total_items < pairs ? p.total_items : pairs);
    p.scalar_a = sA;
    p.scalar_b = sB;
    if (r.variant == 8) {
      if (r.block_n == 64)
        return launch_gemm_2sm_variant<SPG_EPI_LINEAR, 64, 10, false, false, kScaleScalar, true,
                                       true>(maps, p, rr.grid, stream);
      return launch_gemm_2sm_variant<SPG_EPI_LINEAR, 128, 8, false, false, kScaleScalar, true,
                                     true>(maps, p, rr.grid, stream);
    }
    if (r.block_n == 64)
      return launch_gemm_2sm_variant<SPG_EPI_LINEAR, 64, 10, false, false, kScaleScalar, true>(
          maps, p, rr.grid, stream);
    return launch_gemm_2sm_variant<SPG_EPI_LINEAR, 128, 8, false, false, kScaleScalar, true>(
        maps, p, rr.grid, stream);
  }
  const int b_rows = r.block_m == 256 ? r.block_n / 2 : r.block_n;  // B rows staged per CTA
  const bool a_batched = batch > 1 && strideA != 0;
  const bool b_batched = batch > 1 && strideB != 0;
  const int64_t nba = a_batched ? batch : 1, nbb = b_batched ? batch : 1;
  GemmMaps maps;
  bool ok;
  if (a_mn)
    ok = make_tmap_3d(&maps.a, A, false, M, K, nba, M, a_batched ? strideA : M * K, 128, 128, 128);
  else
    ok = make_tmap_3d(&maps.a, A, false, K, M, nba, K, a_batched ? strideA : M * K, 128, 128, 128);
  if (ok) {
    if (b_mn)
      ok = make_tmap_3d(&maps.b, B, false, N, K, nbb, N, b_batched ? strideB : N * K, 128, 128, 128);
    else
      ok = make_tmap_3d(&maps.b, B, false, K, N, nbb, K, b_batched ? strideB : N * K, 128,
                        b_rows, 128);
  }
  if (ok)
    ok = make_tmap_3d(&maps.y, C, true, N, M, batch, N * 2, (batch > 1 ? strideC : M * N) * 2, 32,
                      32, 64);
  if (!ok) return SPG_ERR_CUDA;
  maps.r = maps.y;  // no residual in the per-tensor GEMM
  GemmParams p;
  fill_common_params(p, r, M, N, K, K, N, batch);
  if (!p.err) return SPG_ERR_CUDA;
  if (const spg_status bs = set_bias(p, bias, bias_scale); bs != SPG_OK) return bs;
  // An N-major B half is one 128-byte swizzle row: keep whole tiles there.
  spg_route rr = r;
  if (r.block_m == 256) {
    const int pairs = num_sms() / 2;
    plan_items(p, r, pairs, workspace);
    rr.grid = 2 * (p.total_items < pairs ? p.total_items : pairs);
    if (!b_mn) {
      const uint32_t narrow_rows = static_cast<uint32_t>(r.block_n / p.split_ways / 2);
      if (!make_tmap_3d(&maps.b_narrow, B, false, K, N, nbb, K, b_batched ? strideB : N * K, 128,
                        narrow_rows, 128))
        return SPG_ERR_CUDA;
    } else {
      maps.b_narrow = maps.b;
    }
  }
  p.a_batch_mul = a_batched ? 1 : 0;
  p.b_batch_mul = b_batched ? 1 : 0;
  p.scalar_a = sA;
  p.scalar_b = sB;
  if (!a_mn && !b_mn) return dispatch<false, false>(rr, maps, p, stream);
  if (!a_mn && b_mn) return dispatch<false, true>(rr, maps, p, stream);
  if (a_mn && !b_mn) return dispatch<true, false>(rr, maps, p, stream);
  return dispatch<true, true>(rr, maps, p, stream);
}

}  // namespace

extern "C" spg_status fp8_tensor_gemm(char layout_a, char layout_b, int64_t batch,
                                      const uint8_t* A, int64_t strideA, const float* sA,
                                      const uint8_t* B, int64_t strideB, const float* sB, void* C,
                                      int64_t strideC, int64_t M, int64_t N, int64_t K,
                                      spg_stream_t stream) {
  return tensor_impl(layout_a, layout_b, batch, A, strideA, sA, B, strideB, sB, nullptr, nullptr, C,
                     strideC, M, N, K, nullptr, 0, stream);
}

extern "C" spg_status fp8_tensor_gemm_bias(char layout_a, char layout_b, int64_t batch,
                                           const uint8_t* A, int64_t strideA, const float* sA,
                                           const uint8_t* B, int64_t strideB, const float* sB,
                                           const void* bias, const float* bias_scale, void* C,
                                           int64_t strideC, int64_t M, int64_t N, int64_t K,
                                           spg_stream_t stream) {
  return tensor_impl(layout_a, layout_b, batch, A, strideA, sA, B, strideB, sB, bias, bias_scale,
                     C, strideC, M, N, K, nullptr, 0, stream);
}

extern "C" spg_status fp8_tensor_gemm_ws(char layout_a, char layout_b, int64_t batch,
                                         const uint8_t* A, int64_t strideA, const float* sA,
                                         const uint8_t* B, int64_t strideB, const float* sB,
                                         const void* bias, const float* bias_scale, void* C,
                                         int64_t strideC, int64_t M, int64_t N, int64_t K,
                                         void* workspace, int64_t workspace_bytes,
                                         spg_stream_t stream) {
  return tensor_impl(layout_a, layout_b, batch, A, strideA, sA, B, strideB, sB, bias, bias_scale,
                     C, strideC, M, N, K, workspace, workspace_bytes, stream);
}
