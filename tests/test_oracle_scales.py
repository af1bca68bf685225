"""Pins for the oracle's reading of the cache scales (CPU).

K's scale multiplies the logits and V's scale the output: softmax attention is
invariant to nothing here, so the pins use the two identities linearity gives.
A key scale c equals a softmax scale of c / sqrt(d) on the unscaled keys, and
a value scale c multiplies out by c and leaves lse alone.  A planted swap of
the two scales must fail them.
"""

import math

import numpy as np
import pytest

from oracle import paged_attention as pa

from test_oracle_pins import paged_from_dense, random_requests

SPECS = [(5, 9), (3, 3), (1, 12)]
HQ, HKV, D = 8, 2, 16
TOL = 1e-12


def _run(k_scale=1.0, v_scale=1.0, sm_scale=None, mod=pa, seed=0):
    qs, ks, vs = random_requests(SPECS, HQ, HKV, D, seed=seed)
    args = paged_from_dense(qs, ks, vs, page_size=4, seed=1)
    return mod.paged_prefill(**args, k_scale=k_scale, v_scale=v_scale, sm_scale=sm_scale)


def key_scale_error(mod=pa):
    c = 0.375
    o1, l1 = _run(k_scale=c, mod=mod)
    o2, l2 = _run(sm_scale=c / math.sqrt(D), mod=mod)
    return max(float(np.abs(o1 - o2).max()), float(np.abs(l1 - l2).max()))


def value_scale_error(mod=pa):
    c = 2.5
    o1, l1 = _run(v_scale=c, mod=mod)
    o0, l0 = _run(mod=mod)
    return max(float(np.abs(o1 - c * o0).max()), float(np.abs(l1 - l0).max()))


def test_key_scale_is_a_logit_scale():
    assert key_scale_error() < TOL


def test_value_scale_multiplies_the_output_only():
    assert value_scale_error() < TOL


def test_planted_scale_swap_is_caught(monkeypatch):
    real = pa.paged_prefill

    def swapped(*a, k_scale=1.0, v_scale=1.0, **kw):
        return real(*a, k_scale=v_scale, v_scale=k_scale, **kw)

    monkeypatch.setattr(pa, "paged_prefill", swapped)
    assert max(key_scale_error(), value_scale_error()) > 1e-6
