// Instances of the persistent recurrent kernel for one operator
// (page "Recurrent operators: RNN, GRU, LSTM", Computation).
#include "k_recur.cuh"

namespace rnngb {

cudaError_t launch_recurrent_gru(const RecParams& p, bool exact, int threads, size_t smem,
                                   cudaStream_t stream)
{
    return launch_recurrent_op<1>(p, exact, threads, smem, stream);
}

cudaError_t recurrent_occupancy_gru(int rows_per_thread, bool exact, int threads, size_t smem,
                                      int* blocks)
{
    return recurrent_occupancy_op<1>(rows_per_thread, exact, threads, smem, blocks);
}

}  // namespace rnngb
