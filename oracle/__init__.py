"""CPU oracle for the co-batched layer step — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct fp64 numpy restatement of what one
co-batched transformer layer step computes.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm
may import it; the product path (``co_prefill_decode_gb300``) never does,
and the oracle shares no code with it (only the seeded input generators in
``workload`` serve both).

Sources (page titles):

* ConfluxServe: Reconciling Resource Utilization and Parallelism Efficiency
  across Prefill and Decode in LLM Serving — Fig. 1 (QKV proj -> core
  attention -> O proj -> FFN), §4 and Fig. 7 (prefill and decode tokens
  co-batched through the shared linear operators, attention forked per
  phase), §4 KV residency (decode extends its own KV, prefill appends its
  chunk), App. D Eq. 9 (chunk workload l(c + (l+1)/2)).
* Adaptive Context Parallelism for Production LLM Serving — §2.1
  (Attn = softmax(QK^T/sqrt(d_h) + M) V, M_ij = 0 for j <= i else -inf),
  §2.2 Eq. 1 (W(R, P) = RP + R(R+1)/2).
* Decode Token Parallelism — §4.3 (per layer: rotary embeddings, append the
  new keys/values to the cache, attention; then output projection, residual
  and normalization, MLP), §4.4 Eq. 1 (fused QKV layout, Q then K then V
  heads).

Readings where the pages are silent (each pinned by a test in
``tests/test_oracle.py``): pre-norm residual block with RMSNorm; SwiGLU FFN;
rotate-half RoPE with theta_i = base^(-2i/d); per-head QK-RMSNorm before
RoPE; query head h reads KV head floor(h / G); tensors handed between steps
are bf16 (round-to-nearest-even) while the residual stream h stays at full
precision.

Parity pins: every function here is pinned by a test against something
other than itself (brute force, closed forms, invariants, library routines).
"""
from .layer import (  # noqa: F401
    bf16_round, to_f64, rmsnorm, rope, silu, swiglu, slot_of, gather_request_kv,
    kv_append, attention, decode_attention, prefill_attention, layer_step,
    chunk_workload, LayerWeights64,
)
