"""fp64 CPU oracle of the PrHS sparse-decode path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the test suite, the smoke check
of the package entry file and the CPU-baseline leg of the benchmark import
this package. The CUDA library never calls it and shares no code with it;
both consume the same seeded inputs from ``workloads``.

Every function restates a definition from "Near-Oracle KV Selection via
Pre-hoc Sparsity for Long-Context Inference" (arXiv 2602.08329) and cites the
part of that page it follows. Arithmetic is float64 on inputs widened
exactly from their stored float32/bfloat16 bits.

Pins (tests/test_oracle_pins.py) tie each function to something other than
itself: hand-computed cases, brute force over all subsets on tiny inputs,
closed-form identities, library routines (torch SDPA, scipy cosine) and the
Fig. 4 dilation example. The multi-step CIS schedule (which query is the
anchor, when a fresh retrieval happens) is a reading of Fig. 4 and Fig. 8;
a hand case fixes it where the plausible alternatives part (gating against
the previous query, an anchor query that never moves), and a hand GQA case
fixes which KV head each query head reads (h // G).
"""
from .prhs import (scores, softmax, logsumexp, top_n, dropped_mass, cosine, cis_gate,
                   dilate, dilate_budget, shared_set, attention, dense_attention, decode_head,
                   decode_workload, decode_head_grow, HeadStep, widen)

__all__ = ["scores", "softmax", "logsumexp", "top_n", "dropped_mass", "cosine", "cis_gate",
           "dilate", "dilate_budget", "shared_set", "attention", "dense_attention", "decode_head",
           "decode_workload", "decode_head_grow", "HeadStep", "widen"]
