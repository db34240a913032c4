"""Oracle: a plain, slow CPU restatement of the persistent MoE decode layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The
product path (the CUDA library and its Python binding) never imports, links or
calls anything here, and nothing here imports the product path.

Precision: every contraction and reduction is carried in float64 (numpy), and
values are rounded to bfloat16 exactly at the storage boundaries the layer
defines (round-to-nearest-even).  Where a floating-point value decides an
integer (the NVFP4 codes of an activation, the router's top-k) the decision is
taken in float32, the precision the kernel takes it in.

Sources (page title, section):
  * "Muse Spark Open: 1,109 Tokens a Second Is a Kernel Change, Not a Model
    Change" (orcarouter.ai), section "Where the kernel boundary sits, and why it
    stops there": launch boundary (attention through next QKV + KV write), GQA
    with a 2,048-token sliding window or global attention, routing to 8 of 256
    experts, NVFP4 experts, pooler/unpooler, fp4 after the first expert GEMM and
    bf16 after the second.
  * same page, section "What the 5.9 ms is still spent on": the combine of
    the expert outputs.
  * The pages name neither the norm, its epsilon, positional encoding, the
    router's normalisation nor the activation quantisation.  Each function
    states the plain reading it takes (RMSNorm with eps 1e-6, no RoPE,
    softmax-then-top-k without renormalisation, per-row NVFP4 quantisation of
    the expert inputs).

Parity status: every function here is pinned by tests/test_oracle_*.py against
library routines (torch's float8/bfloat16/float16 casts, numpy sorts), closed
forms, invariants and brute force on tiny inputs.  The whole-layer composition
on trained weights has no printed values to pin to: "parity unpinned" for
real-model numerics, since the pages print no worked example.
"""

from . import numerics, layer  # noqa: F401
