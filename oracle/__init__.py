"""CPU oracle for the flow-matching action-expert denoise loop.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (the CUDA library and its Python binding) never calls it and shares no
code with it; the only code both sides use is the seeded input generator in
``synth``, which holds none of the method's arithmetic.

The oracle is plain numpy in float64 by default (``dtype=np.float32`` gives
an fp32 instantiation).  Every function follows one passage of the source
pages, cited in its docstring as "<page title>, <section / equation>":

* "vla.cpp: A Unified Inference Runtime for Vision-Language-Action Models"
  (arXiv 2606.08094v2): Eq. (1) Euler integration, Eq. (2) attention,
  Eq. (5) error metrics.
* "pi0.5 Design" (TensorRT Edge-LLM developer guide): the action expert
  geometry, the hoisted ``cond`` component, the modulation-row layout
  (Component contract), attention over prefix ++ own K/V (Attention and the
  K/V pool).
* "GR00T N1.7" (TensorRT Edge-LLM developer guide): the action component,
  the hoisted AdaLN table and ``action_time_bias`` (Build-time constants).
* "Optimizing GR00T-N1.7 Training" (LoongForge blog, section 3.3): the
  rotate-half RoPE convention.

Where the pages are silent the oracle takes one documented reading; each is
listed in the repository's design notes (readings S1-S14).

Pins: every function is checked in ``tests/test_oracle_pins.py`` against
closed forms, invariants, library routines (torch CPU) or brute force.
"""
from .ops import (gelu_tanh, swish, rms_norm, layer_norm, rope_rotate_half, e4m3_decode, dequantize_rows,
                  attention, error_metrics)
from .schedule import schedule, euler, time_embedding, time_condition, modulation_table
from .expert import expert_velocity, expert_denoise
from .dit import dit_velocity, dit_denoise, action_time_bias, project_context, encode_state
from .denoise import denoise, velocity

__all__ = [
    "gelu_tanh", "swish", "rms_norm", "layer_norm", "rope_rotate_half",
    "attention", "error_metrics", "schedule", "time_embedding",
    "time_condition", "modulation_table", "expert_velocity", "expert_denoise",
    "dit_velocity", "dit_denoise", "action_time_bias", "denoise", "velocity",
    "euler", "e4m3_decode", "dequantize_rows", "project_context", "encode_state",
]
