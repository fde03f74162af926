// qmv_q4k.cu -- Q4_K instances of the decode mat-vec (batch 1..8, plus the recording variant).
#include "qmv.cuh"

namespace qmd {

qmd_status launch_qmv_q4k(const QmvArgs &a, const QmvPlan &plan, cudaStream_t s)
{
    return launch_qmv<false>(a, plan, s);
}

}  // namespace qmd
