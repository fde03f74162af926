// qmv_q6k.cu -- Q6_K (split layout) instances of the decode mat-vec (batch 1..8, plus the
// recording variant).
#include "qmv.cuh"

namespace qmd {

qmd_status launch_qmv_q6k(const QmvArgs &a, const QmvPlan &plan, cudaStream_t s)
{
    return launch_qmv<true>(a, plan, s);
}

}  // namespace qmd
