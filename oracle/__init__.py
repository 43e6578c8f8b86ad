"""fp64 CPU oracle for the forward pass of one Hy3-style MoE FFN layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path (no kernels, headers, helpers or tables) and never
takes an input or an expected value from it.

Every function is a plain restatement, in float64 numpy, of what the pages
define; matrix products use ``numpy.matmul`` as a library primitive, nothing is
blocked, fused or reordered.  Sources (by page title and section):

* hy3 README ("hy3 -- tencent/Hy3 GGUF Converter and Inference Engine"),
  "Model facts" table, row "MoE routing": sigmoid of the router logits, top-8
  chosen on sigmoid + expert_bias, combine weights are the unbiased sigmoids
  renormalised to sum 1 and scaled by router_scaling_factor = 2.826; one
  always-active shared expert; expert intermediate size 1536.
* "Hy3 Preview inference optimisation case" (llm-wiki digest), section 2
  "Router GEMM": the fp32 router weight is split offline as
  W ~ W_high + scale * W_low with scale = 1/256, two BF16 GEMMs, two
  accumulators, one FFMA in the epilogue.  Section 3 "FusedMoE": routing and
  index preprocessing that reserves one contiguous output range per expert;
  gate-up GEMM reading the original input through the route index; down GEMM
  written compactly per expert; top-k weighted aggregation at the end.
* "HunyuanImage 3.0 MoE reading" post, sections "HunyuanTopKGate easy_topk",
  "Routed Experts" and "Shared MLP": the fp32 router Linear (no bias), softmax
  over experts, top-k, division by clamp(sum, min=1e-8); the eager path that
  flattens topk_idx, repeats each token k times, runs each expert on the rows
  routed to it, multiplies by the top-k weights and sums over k; the shared
  MLP as a parallel branch added to the routed output; SwiGLU experts
  down(SiLU(gate(x)) * up(x)).

Readings where the pages are silent (each also listed in the design notes):

* the split: W_high = bf16_RNE(W), W_low = bf16_RNE((W - W_high) * 256);
* top-k order: descending key, equal keys go to the lower expert index;
* no epsilon in the sigmoid renormalisation; route_scale does not touch the
  shared expert; the shared expert is ungated and has intermediate size I;
* the order of slots inside an expert segment is ascending flat slot t*k + j;
* FP8 expert weights (the Hy3 case's W8A8 deployments, format unspecified):
  OCP E4M3 codes with one fp32 scale per output row, max|row| / 448, rounded
  to nearest-even and saturated at 448; the layer uses value * scale.
* W8A8 (the case's "activation quantisation + Down GEMM"): every activation
  matrix feeding an expert GEMM is quantised per row by the same rule, from its
  own values -- the hidden state per token, the bf16 SiLU(gate) * up activation
  per routed slot; the router stays fp32.
* MXFP8 / MXFP4 (the Ascend deployment article, section 8.2, names them and
  no more): the OCP Microscaling formats, blocks of 32 along the reduction axis
  with a power-of-two scale 2^(floor(log2 max) - emax), E4M3 or E2M1 elements
  nearest-even and saturated (``oracle/mx.py``; the article's hybrid: MXFP4
  routed weights, MXFP8 shared weights and activations).

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, hand-worked examples (``tests/golden/``), brute force on
tiny inputs, or textbook reductions.  Nothing here is "parity unpinned".
"""
from .moe import (  # noqa: F401
    widen_bf16,
    bf16_round,
    router_logits,
    split_router_weight,
    router_logits_split,
    sigmoid,
    silu,
    topk_desc,
    route_sigmoid,
    route_softmax,
    renormalize,
    routing_weights_for,
    near_tie_alternatives,
    histogram_offsets,
    permutation,
    swiglu,
    expert_outputs_sorted,
    shared_expert,
    combine,
    layer_forward,
    layer_rows,
    e4m3_value,
    e4m3_encode,
    quantize_rows_e4m3,
    dequantize_rows_e4m3,
    quantized_matmul,
    swiglu_w8a8,
    layer_forward_w8a8,
)
