"""CPU checks of the synthetic input recipe against the trace figures ConfluxServe reports.

The decode-heavy mix stands in for the Mooncake Toolagent trace, whose prompt
lengths ConfluxServe §8 (Table 3) reports as P50 6,346 and P95 26,114
tokens.  The recipe draws clip(rint(exp(N(ln 6346, 0.86))), 512, 32768):
0.86 = ln(26114 / 6346) / 1.645 puts the log-normal's 95th percentile on the
trace's."""
import math

import numpy as np
import torch

import workload as wl

P50, P95 = 6346, 26114          # Table 3, Mooncake Toolagent prompt lengths


def test_sigma_puts_the_95th_percentile_on_the_trace():
    med, sigma, lo, hi = wl.WORKLOADS["mix"].lognormal
    assert med == P50
    assert abs(med * math.exp(1.6448536 * sigma) - P95) / P95 < 2e-3
    assert lo <= P50 and P95 <= hi            # the clip leaves both quantiles alone


def test_drawn_lengths_match_the_trace_quantiles():
    w = wl.WORKLOADS["mix"]
    g = torch.Generator().manual_seed(123)
    x = wl._lognormal_lengths(w, 200_000, g)
    assert x.min() >= 512 and x.max() <= 32768
    q50, q95 = np.quantile(x, [0.5, 0.95])
    assert abs(q50 - P50) / P50 < 0.02
    assert abs(q95 - P95) / P95 < 0.03


def test_mix_batch_draws_its_contexts_from_the_recipe():
    w = wl.WORKLOADS["mix"]
    b = wl.make_batch(w, 0)
    assert b.n_decode == 128 and b.prefill_len == 256
    ctx = np.asarray(b.dec_ctx)
    assert ctx.min() >= 512 and ctx.max() <= 32768 and 512 <= b.prefill_prefix <= 32768
    # seeded: the same batch every time
    b2 = wl.make_batch(w, 0)
    assert np.array_equal(ctx, np.asarray(b2.dec_ctx)) and b.prefill_prefix == b2.prefill_prefix
