// Decode-shaped (swapped operand) instantiations of KIND_GATE_UP: A = weight rows,
// B = the step's tokens (N = 16 .. 128).
#include "gemm_launch.cuh"

namespace tpl {

cudaError_t launch_gemm_decode_gate_up(int bn, const CUtensorMap& a, const CUtensorMap& w,
                                  const GemmParams& p, int grid, cudaStream_t st) {
  switch (bn) {
    case 16: return launch_one<true, KIND_GATE_UP, 16, 2>(a, w, p, grid, st);
    case 32: return launch_one<true, KIND_GATE_UP, 32, 2>(a, w, p, grid, st);
    case 64: return launch_one<true, KIND_GATE_UP, 64, 2>(a, w, p, grid, st);
    case 128: return launch_one<true, KIND_GATE_UP, 128, 2>(a, w, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

int gemm_stages_decode_gate_up(int bn) {
  switch (bn) {
    case 16: return GemmShape<true, KIND_GATE_UP, 16, 2>::kStages;
    case 32: return GemmShape<true, KIND_GATE_UP, 32, 2>::kStages;
    case 64: return GemmShape<true, KIND_GATE_UP, 64, 2>::kStages;
    case 128: return GemmShape<true, KIND_GATE_UP, 128, 2>::kStages;
    default: return 0;
  }
}

}  // namespace tpl
