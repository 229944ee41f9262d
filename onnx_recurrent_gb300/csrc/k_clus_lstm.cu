// Instances of the dataflow kernel with the in-cluster exchange of h for one
// operator (page "Recurrent operators: RNN, GRU, LSTM", Computation).
#include "k_recur2.cuh"

namespace rnngb {

cudaError_t launch_cluster_lstm(const RecParams& p, bool exact, int threads, size_t smem, cudaStream_t stream)
{
    return launch_cluster_op<2>(p, exact, threads, smem, stream);
}

cudaError_t cluster_occupancy_lstm(int tn, bool exact, bool two, int ctas, int cluster, int threads, size_t smem,
                                  int* clusters)
{
    return cluster_occupancy_op<2>(tn, exact, two, ctas, cluster, threads, smem, clusters);
}

}  // namespace rnngb
