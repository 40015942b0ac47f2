"""CPU oracle of block-cached, confidence-threshold masked-diffusion decoding.

TEST INFRASTRUCTURE, not part of the product.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg
import it.  It shares no code with the CUDA path: it reads its inputs from
``cached_masked_decoding_gb300.synth`` (the seeded generator, which holds none of
the method's arithmetic) and nothing else from the package.

Precision: float64 throughout (numpy; matrix products through BLAS), weights
widened exactly from their bf16 bits.  Where a floating-point value decides an
integer (threshold, fallback, top-k, factor rule) the decision is taken in
float32 on the confidence rounded to float32, the precision the GPU kernel
decides in.

Parity status of each function is stated in its module header.
"""
from . import model, sampler, theory  # noqa: F401
