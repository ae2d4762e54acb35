"""CPU oracle for the looped normalized-GPT forward pass.

TEST INFRASTRUCTURE: a plain, slow numpy implementation that the CUDA path
is checked against.  It shares no code with the CUDA library.  Only the
tests, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` may
import it; the product path never does.

Parity status of each function is listed in oracle/model.py and the pins
that anchor it are in tests/test_oracle_pins.py.  Quantisation
(oracle/quant.py), sampling (oracle/sampling.py) and the truncated-
backpropagation training step (oracle/train.py, torch float64) have their
own pin files.
"""
from .model import (LAST_LOOP, PER_LOOP, Oracle, Trace, attention, kv_bytes, l2n,
                    loop_schedule, ngpt_update, rope, silu, sigmoid, slot_positions)

__all__ = ["LAST_LOOP", "PER_LOOP", "Oracle", "Trace", "attention", "kv_bytes", "l2n",
           "loop_schedule", "ngpt_update", "rope", "silu", "sigmoid", "slot_positions"]
