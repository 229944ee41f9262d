// Instances of the persistent recurrent kernels for one operator
// (page "Recurrent operators: RNN, GRU, LSTM", Computation).
#include "k_recur.cuh"
#include "k_recur2.cuh"

namespace rnngb {

cudaError_t launch_recurrent_lstm(const RecParams& p, bool exact, int threads, size_t smem,
                                   cudaStream_t stream)
{
    if (p.kernel == 2) return launch_dataflow_op<2>(p, exact, threads, smem, stream);
    return launch_recurrent_op<2>(p, exact, threads, smem, stream);
}

cudaError_t recurrent_occupancy_lstm(int kernel, int lbr, int rows_per_thread, int gs, bool exact, int threads,
                                      size_t smem, int* blocks)
{
    if (kernel == 2) return dataflow_occupancy_op<2>(rows_per_thread, exact, false, gs, threads, smem, blocks);
    return recurrent_occupancy_op<2>(rows_per_thread, exact, threads, smem, blocks);
}

}  // namespace rnngb
