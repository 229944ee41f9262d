"""GB300 (sm_103a) ONNX RNN / GRU / LSTM sequence operator.

The operator lives in a CUDA library with a C ABI (include/onnx_recurrent.h);
``rnn`` is its ctypes binding and ``synth`` draws seeded synthetic inputs.
"""
from ._build import build
from .rnn import (Plan, RNNError, Stack, rnn_stack_create, rnn_stack_destroy, rnn_stack_last_launch_count,
                  rnn_stack_last_wavefront, rnn_stack_run, rnn_stack_set_wavefront, load, rnn_cell_plan_create, rnn_cell_run, rnn_last_error, rnn_plan_create, rnn_plan_debug_barrier,
                  rnn_plan_destroy, rnn_plan_get_activation, rnn_plan_get_launch,
                  rnn_plan_last_launch_count, rnn_plan_last_timing, rnn_plan_set_launch,
                  rnn_plan_timing_totals,
                  rnn_plan_set_io_type, rnn_plan_set_mode, rnn_plan_set_timing, rnn_plan_set_weights, rnn_plan_sync,
                  rnn_run, run)

__all__ = ["build", "load", "Plan", "RNNError", "rnn_plan_create", "rnn_run", "rnn_plan_destroy",
           "rnn_plan_set_mode", "rnn_plan_set_weights", "rnn_plan_sync", "rnn_plan_get_activation",
           "rnn_plan_set_launch", "rnn_plan_get_launch", "rnn_plan_set_timing",
           "rnn_plan_last_timing", "rnn_plan_timing_totals", "rnn_plan_debug_barrier", "rnn_plan_last_launch_count",
           "rnn_last_error", "rnn_cell_plan_create", "rnn_cell_run", "rnn_plan_set_io_type", "Stack", "rnn_stack_create", "rnn_stack_run", "rnn_stack_destroy",
           "rnn_stack_last_launch_count", "rnn_stack_set_wavefront", "rnn_stack_last_wavefront", "run"]
