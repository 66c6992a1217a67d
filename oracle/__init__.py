"""Plain, slow, fp64 CPU oracle for the decode GEMV with a fused epilogue and the
signed Walsh-Hadamard prologue.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or run this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` use it.  It shares no code with the CUDA library (no kernels, headers,
helpers, tables or constant generators) and it imports nothing from the product
package.  Its inputs come from the caller (in the tests: the seeded generators in
``decode_gemv_epilogue_gb300.synth``, which hold none of the method's arithmetic).

Sources, cited by page title and section:

* [EPI]  "feat(cuda): fuse activations and residual add into mmv f/q epilogues"
         -- Summary; What changed (the three fused tails); Why.
* [FWHT] "vulkan: fuse the sign multiply into the Hadamard FWHT" -- Overview
         (MUL(signs) -> RESHAPE -> MUL_MAT(hint=hadamard); sign applied while the row
         is loaded, before the transform; sign vector broadcast over its length).
* [CPU]  "ggml-cpu: fuse element-wise epilogues (ADD, MUL, SILU) into
         ggml_compute_forward_mul_mat" -- What (fused pairs table), Guards, Correctness
         (F32 / F16 / Q8_0 / Q4_0 weights; fusion leaves the values unchanged).

Everything is computed in float64 from the stored weight bytes.  The method is an
exact re-arrangement of a plain computation (the fused tail reads the same values the
separate passes would), so the oracle is that plain computation written out:
dequantise -> dot product -> element-wise tail, and x' = H.(x*s)/sqrt(B) per block.

Parity status of every function is listed in ``PINS`` below; each one is pinned by
``tests/test_oracle_pins.py`` to closed forms, printed fixtures under
``tests/golden/``, library special cases or brute force, never to itself.
"""

from . import quant, gemv, fwht, chain, norm  # noqa: F401

PINS = {
    "quant.dequantize_f32": "pinned: bit pattern fixture, identity",
    "quant.dequantize_f16": "pinned: hand-decoded binary16 fixture + numpy float16 (library)",
    "quant.dequantize_q8_0": "pinned: hand-decoded block fixture (golden/q8_0_block.txt)",
    "quant.dequantize_q4_0": "pinned: hand-decoded block fixture (golden/q4_0_block.txt)",
    "quant.dequantize_q4_k": "pinned: hand-packed super-block (golden/q4_k_block.txt), zero codes / zero dmin, "
                             "random fields through the generator's packer",
    "gemv.gemv": "pinned: 2x3 worked integer example, identity W, one-hot x, brute force",
    "gemv.apply_epilogue": "pinned: sigmoid(0)=1/2, silu(0)=0, symmetry, limits, W=0 cases",
    "fwht.hadamard": "pinned: H2, Sylvester recursion via np.kron, scipy.linalg.hadamard, H.H=nI",
    "fwht.fwht_signed": "pinned: butterfly vs dense, e0 -> 1/sqrt(B), ones -> sqrt(B) e0, Parseval, involution",
    "chain.decode_layer": "pinned: composition on identity-like tiny weights (closed form)",
    "gemv.gemv_glu": "pinned: hand-worked 3x2 example (golden/glu_worked.txt), zero gate/up, one-hot x",
    "norm.rms_norm": "pinned: hand-worked example (golden/rms_norm_worked.txt), unit mean square, "
                     "scale invariance, constant input, eps-dominated limit",
}
