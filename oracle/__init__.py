"""CPU oracle for the DSA indexer (test infrastructure, not the product).

A plain, slow, obviously correct restatement of what the indexer computes,
written from the four pages on the bf16 index-K fix in the DSA indexer:

  * "The Moment of Validation: Diagnosing an OOM Crash in the bf16 Index-K Fix
    for DeepSeek V4 Sparse Attention" (section "Input Knowledge Required to
    Understand This Message": 128 e4m3 bytes + a 4-byte scale = 132 B/token for
    fp8, 128 x 2 B = 256 B/token for bf16; the fused store does normalisation,
    RoPE and the store in one pass);
  * "The Fused Kernel Decision: Precision Archaeology in the CUDA Sparse
    Attention Indexer" (section "The Message": a paged bf16 index cache of
    64-token pages laid out [npages, 64*128]; a token maps to a page and an
    offset within it);
  * "The Crash That Changed Direction" (sections "The Experiment: Why fp32?"
    and "Assumptions Made and Broken": the indexer scores keys with a batched
    matrix product followed by a ReLU, up-converts fp8 keys exactly before the
    product, and keeps the top-K positions; K is 512, raised to 1024);
  * "When the Fused Kernel Isn't Enough" (section "The Message: Validation and
    Discovery": materialising the logits over the whole context is what ran
    out of memory).

Where the pages leave a step open, the oracle takes the plainest reading:
per-head ReLU, a head-weighted sum over the 64 heads, causal masking, ties
broken toward the lower position, RoPE pairing dims i and i+64 (half-split),
RNE rounding everywhere and e4m3 saturating at +-448.

Only tests/, __graft_entry__.smoke() and bench.py (its CPU-baseline and
reference legs) may import this package. The GPU library never calls it and
shares no code with it.

Modules:
  formats  - bf16 and OCP FP8 E4M3 encode/decode from the formats' definitions
  store    - RMSNorm + RoPE + quantise + paged write, fp32 with a fixed order
  indexer  - scores in float64 and exact top-k by (score desc, position asc)
"""
