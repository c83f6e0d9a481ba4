// Decode-shaped (swapped operand) instantiations of KIND_GATE_UP: A = 256 weight
// rows, B = the step's tokens (N = 16 .. 128).
#include "gemm_launch.cuh"

namespace tpl {

cudaError_t launch_gemm_decode_gate_up(int bn, const CUtensorMap& a, const GemmParams& p, int grid,
                                  cudaStream_t st) {
  switch (bn) {
    case 16: return launch_one<true, KIND_GATE_UP, 16>(a, p, grid, st);
    case 32: return launch_one<true, KIND_GATE_UP, 32>(a, p, grid, st);
    case 64: return launch_one<true, KIND_GATE_UP, 64>(a, p, grid, st);
    case 128: return launch_one<true, KIND_GATE_UP, 128>(a, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

int gemm_stages_decode_gate_up(int bn) {
  switch (bn) {
    case 16: return GemmShape<true, KIND_GATE_UP, 16>::kStages;
    case 32: return GemmShape<true, KIND_GATE_UP, 32>::kStages;
    case 64: return GemmShape<true, KIND_GATE_UP, 64>::kStages;
    case 128: return GemmShape<true, KIND_GATE_UP, 128>::kStages;
    default: return 0;
  }
}

}  // namespace tpl
