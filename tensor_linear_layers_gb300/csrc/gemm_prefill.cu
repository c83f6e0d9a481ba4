// Prefill-shaped instantiations: A = 128 tokens, B = 256 weight rows.
#include "gemm_launch.cuh"

namespace tpl {

cudaError_t launch_gemm_prefill(int kind, const CUtensorMap& a, const GemmParams& p, int grid,
                                cudaStream_t st) {
  switch (kind) {
    case KIND_GATE_UP: return launch_one<false, KIND_GATE_UP, 256>(a, p, grid, st);
    case KIND_COL: return launch_one<false, KIND_COL, 256>(a, p, grid, st);
    case KIND_ROW: return launch_one<false, KIND_ROW, 256>(a, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

// QKV (column-parallel) and o_proj (row-parallel) of one attention block are
// independent: one launch walks both problems' tiles.
cudaError_t launch_gemm_prefill_col_row(const CUtensorMap& a1, const GemmParams& p1, const CUtensorMap& a2,
                                        const GemmParams& p2, int grid, cudaStream_t st) {
  return launch_one<false, KIND_COL, 256, KIND_ROW>(a1, p1, grid, st, &a2, &p2);
}

int gemm_stages_prefill(int kind) {
  switch (kind) {
    case KIND_GATE_UP: return GemmShape<false, KIND_GATE_UP, 256>::kStages;
    case KIND_COL: return GemmShape<false, KIND_COL, 256>::kStages;
    case KIND_ROW: return GemmShape<false, KIND_ROW, 256>::kStages;
    default: return 0;
  }
}

}  // namespace tpl
