"""fp64 CPU oracle for the MXFP4 mixture-of-experts layer — TEST INFRASTRUCTURE.

Plain, slow, obviously correct reference arithmetic. Only the test suite,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs
of ``bench.py`` may import or run anything in this package. The product path
(the CUDA library and its Python binding) never imports it, and this package
imports nothing from the product path: the two share no code. Both sides get
their inputs from the separate ``workloads`` module.

Contents
  mxfp4  — E2M1/E8M0 decode and the MX quantisation rule (pack oracle)
  moe    — router logits, top-k + renormalised softmax, expert SwiGLU,
           shared expert, layer output, and the token->expert sort
  mxfp8  — E4M3 activation quantisation for the W4A8 mode
  lmhead — the FP8 (per-row scale) LM-head GEMV

Pin status of every function is listed in the module docstrings; none is
"parity unpinned".
"""
from . import lmhead, mxfp4, moe, mxfp8  # noqa: F401
