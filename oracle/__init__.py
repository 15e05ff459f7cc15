"""Float64 CPU oracle for the multi-LoRA decode hot path.

TEST INFRASTRUCTURE ONLY.  This package states, plainly and slowly, what the
hot path computes, so the CUDA library can be checked against it.  Only the
test suite, the smoke check (``__graft_entry__.smoke``) and the CPU-baseline
leg of ``bench.py`` may import it.  The product path (the C-ABI library and its
Python binding) never imports, calls or links anything here, and this package
never imports the product.  The two share only the seeded input generators in
``workloads``, which hold none of the method's arithmetic.

Sources:
  * "Multi-LoRA Serving in Practice: Serving Multiple Business Adapters with
    One Base Model", section "Core Principle: Shared Base Model, Per-Request
    Adapter Selection": the LoRA layer output = W·x + scale · B(A·x), with the
    adapter chosen per request.
  * "LoRA Inference" (glossary), weight-merging paragraph: the merged weight
    W = W0 + ΔW gives the same layer output (used as a pin, not as the oracle).
  * "InvisibleLoRA: Fast Multi-LoRA Serving Without Per-Token LoRA Decoding",
    abstract: a LoRA-off pass drafts, one LoRA-on pass verifies every draft,
    and verification keeps the output distribution of plain multi-LoRA
    decoding.  The pages give no accept rule; the oracle takes standard
    speculative sampling (Leviathan, Kalman & Matias 2023; Chen et al. 2023)
    with an exact fixed-point residual draw (see ``oracle.accept``).

Modules: ``oracle.layer`` (segment plan, shrink, layer output),
``oracle.accept`` (accept test, residual/bonus sample), ``oracle.softmax``
(logits to probabilities, draft-token draw), ``oracle.gate`` (the run-time
draft gate's cost model), ``oracle.kvcache`` (where each pass's K/V rows
go in the paged cache the two passes share) and ``oracle.fp8`` (E4M3
rounding, per-row scales and the draft layer on FP8 weights).  Every function is pinned by
tests under ``-m "not gpu"``; none is marked "parity unpinned".
"""
