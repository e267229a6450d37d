"""FP64 CPU oracle of the routed block-scaled FP4 mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code, table or constant generator with
the CUDA library; both sides draw their inputs from ``synth``.

Modules, each written from the pages' description of the method:

* ``formats``  - E2M1, E8M0 and E4M3 decoding and round-to-nearest-even encoding.
* ``quant``    - MXFP4 (E8M0 per 32) and NVFP4 (E4M3 per 16 + FP32 tensor scale)
                 quantisation of activations.
* ``router``   - sigmoid + correction-bias grouped top-k routing.
* ``permute``  - expert histogram and stable token permutation.
* ``moe``      - expert MLP (gate/up, SwiGLU, requantised intermediate, down),
                 weighted combine, and the output tolerance with its ambiguity
                 allowance.
* ``convert``  - exact MXFP4 -> FP8 E4M3 per-channel conversion.

Every function is pinned by the CPU tests in ``tests/test_oracle_*.py`` against
closed forms, library routines, brute force or invariants.
"""
from . import formats, quant, router, permute, moe, convert  # noqa: F401
