"""CPU oracle for the block-quantized MoE layer and greedy MTP acceptance.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
legs of ``bench.py`` may use it.  It shares no code with the CUDA path.

Everything here is plain numpy.  Block formats are decoded to fp32 exactly as
defined in :mod:`oracle.formats`; routing, the expert FFNs and the combine run
in fp64 (:mod:`oracle.moe`); acceptance is :mod:`oracle.accept`; one MTP
draft/verify round (target stack, output norm, LM head, draft heads,
acceptance) is :mod:`oracle.mtp`.

Sources (page title, section):
  * "Step-5 Preview GGUF" (smalinin/Step-5-Preview-GGUF), "Model background"
    configuration table: hidden 4096, 352 routed experts with 8 selected per
    token; "Precision distribution" table: routed experts in low-bit block
    types, shared experts and the output matrix in Q8_0, routers in F32.
  * "Step 3.7 Flash Mixed-Quant GGUF", "Tensor recipe" table: routed experts
    in Q4_K, shared experts in Q8_0, router F32.
  * "Support Step3.5/3.7 flash mtp3" (llama.cpp PR #24340), "Overview"
    data-flow trace, Round 1 steps (1) target batch of id_last plus three
    drafts, (4) verify, (5) accept.

The pages name Q8_0 / Q4_K and a softmax-free "router" only by name; the
arithmetic of the formats, of the router (softmax over all experts, top-k,
renormalise, ties to the lower expert index) and of the SwiGLU experts is the
plainest reading of the layer those pages describe.  Each reading is stated
where it is used.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(hand-built blocks, brute force on tiny inputs, closed forms, the PR's worked
acceptance example).  The end-to-end layer values themselves have no printed
counterpart on the pages: they are pinned only through those parts.
"""

from . import formats, moe, accept, mtp  # noqa: F401
