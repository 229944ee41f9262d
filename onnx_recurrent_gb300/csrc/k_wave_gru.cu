// Instances of the stacked-layer wavefront kernel for one operator
// (page "Recurrent operators: RNN, GRU, LSTM", Computation).
#include "k_wave.cuh"

namespace rnngb {

cudaError_t launch_wavefront_gru(const WaveParams& p, bool exact, int tn, int ctas, int threads, size_t smem,
                                   cudaStream_t stream)
{
    return launch_wavefront_op<1>(p, exact, tn, ctas, threads, smem, stream);
}

cudaError_t wavefront_occupancy_gru(int tn, bool exact, int threads, size_t smem, int* blocks)
{
    return wavefront_occupancy_op<1>(tn, exact, threads, smem, blocks);
}

}  // namespace rnngb
