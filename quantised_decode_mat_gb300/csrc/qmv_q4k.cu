// qmv_q4k.cu -- Q4_K instances of the decode mat-vec (batch 1..8, plus the recording variant).
#include "qmv_splitk.cuh"

namespace qmd {

qmd_status launch_qmv_q4k(const QmvArgs &a, const QmvPlan &plan, cudaStream_t s)
{
    QmvKParams kp;
    int mode = QMV_PLAIN;
    const qmd_status st = make_params(a, plan, kp, mode);
    if (st != QMD_OK)
        return st;
    if (plan.layout == 1)
        return launch_qmv_tc<QMD_Q4_K>(kp, plan, mode, s);
    if (plan.layout == 2)
        return launch_qmv_rl<QMD_Q4_K>(kp, plan, mode, a.batch, s);
    if (plan.layout == 3)
        return launch_qmv_sk<QMD_Q4_K>(kp, plan, mode, a.batch, s);
    return launch_qmv_slice<QMD_Q4_K>(kp, plan, a.batch, mode, s);
}

int qmv_regs_q4k(int batch, int PR, int mode) { return qmv_slice_regs<QMD_Q4_K>(batch, PR, mode); }

}  // namespace qmd
