"""CPU oracle for the SubSpec draft-and-verify decode step.

TEST INFRASTRUCTURE ONLY.  Plain, slow, obviously-correct NumPy code that
states what the decode step computes, used to check the CUDA library.  Only
`tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` may
import it; the library never does, and it imports nothing from the library.

Sources (the three pages on SubSpec):
  * "SubSpec: Using the Target Model's Own Low-Bit Shadow as Its Draft Model"
    (a reading report; cited as "Low-Bit Shadow report", with its section);
  * "Speculate Deep and Accurate: Lossless and Training-Free Acceleration for
    Offloaded LLMs via Substitute Speculative Decoding", the summary card
    (cited as "Speculate Deep and Accurate card", with its heading);
  * the same title's citation-map entry with the arXiv abstract (cited as
    "Speculate Deep and Accurate abstract").

Precision: activations fp32, weights exact bf16 values, every matrix product
accumulated in float64 and rounded to fp32, softmax / log-softmax / logsumexp
in float64.  The tensors a bf16 decoder stores in bf16 (matrix-product inputs,
the KV cache, the attention output) are rounded to bf16 with ties-to-even.

Modules:
  bf16     -- rounding helpers
  quant    -- group-64 min-max int4 pack / dequant / W4 product
  philox   -- Philox4x32-10 counter-based generator and Gumbel noise
  model    -- the decoder forward over rows with an explicit visibility mask
  tree     -- draft-tree expansion, accept walk, tree attention by path
  decode   -- plain decoding, SubSpec decoding, teacher-forced stream check

Every function is pinned by a `-m "not gpu"` test against something other
than itself (closed forms, published test vectors, brute force, invariants).
"""
