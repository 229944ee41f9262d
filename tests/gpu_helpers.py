"""Run an RNNCase through the CUDA library (C ABI via the binding)."""
import numpy as np

import onnx_recurrent_gb300 as orc


def to_dev(a, torch):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_case(case, mode="exact", launch=None, const_weights=False, want=("Y", "Y_h", "Y_c"),
             plan=None, keep_plan=False):
    import torch
    own = plan is None
    if own:
        plan = orc.rnn_plan_create(case.op, case.direction, case.hidden_size, case.input_size,
                                   activations=case.activations, alpha=case.alpha, beta=case.beta,
                                   clip=case.clip, layout=case.layout,
                                   linear_before_reset=case.linear_before_reset,
                                   input_forget=case.input_forget)
        orc.rnn_plan_set_mode(plan, mode)
        if launch:
            orc.rnn_plan_set_launch(plan, *launch)
    t = {k: to_dev(v, torch) for k, v in case.tensors().items()}
    W, R = t["W"], t["R"]
    if const_weights:
        orc.rnn_plan_set_weights(plan, W, R)
        W = R = None
    Y = torch.full(case.y_shape(), float("nan"), device="cuda") if "Y" in want else None
    Yh = torch.full(case.state_shape(), float("nan"), device="cuda") if "Y_h" in want else None
    Yc = (torch.full(case.state_shape(), float("nan"), device="cuda")
          if ("Y_c" in want and case.op == "LSTM") else None)
    if const_weights:
        # W/R are ignored once constant; pass them as NULL through the C ABI
        st = orc.load().rnn_run(plan.handle, case.seq, case.batch, orc.rnn._ptr(t["X"]), None, None,
                                orc.rnn._ptr(t["B"]), orc.rnn._ptr(t["sequence_lens"]),
                                orc.rnn._ptr(t["initial_h"]), orc.rnn._ptr(t["initial_c"]),
                                orc.rnn._ptr(t["P"]), orc.rnn._ptr(Y), orc.rnn._ptr(Yh),
                                orc.rnn._ptr(Yc), orc.rnn._stream(None))
        orc.rnn._check(st)
    else:
        orc.rnn_run(plan, t["X"], W, R, t["B"], t["sequence_lens"], t["initial_h"],
                    t["initial_c"], t["P"], Y, Yh, Yc)
    orc.rnn_plan_sync(plan)
    torch.cuda.synchronize()
    out = tuple(None if v is None else v.cpu().numpy() for v in (Y, Yh, Yc))
    if own and not keep_plan:
        orc.rnn_plan_destroy(plan)
        return out
    return out + (plan,) if keep_plan else out


def row_slice(case, rows, arr, kind):
    """Select batch rows of an output array (kind 'Y' or 'state')."""
    rows = list(rows)
    if arr is None:
        return None
    if case.layout == 1:
        return arr[rows]
    return arr[:, :, rows] if kind == "Y" else arr[:, rows]
