"""Plant plausible mistakes in the oracle (CPU only) and check that the pins notice them.

Each mutant replaces the oracle's per-sequence attention kernel with a variant carrying one
mistake: a dropped softmax scale, the wrong GQA head mapping, keys and values swapped, or a
causal window that leaves out the query's own key.  The comparison with torch's
scaled_dot_product_attention (the pin of the contiguous special case) must fail for every
mutant and pass for the real oracle.
"""

import numpy as np
import pytest

import oracle.paged_kv as pa
from synthetic import make_workload
from test_oracle_attention import _attn, _pools, _sdpa_seq

_real = pa._attend


def _mut_no_scale(q, K, V, first, scale, group):
    return _real(q, K, V, first, 1.0, group)


def _mut_gqa_modulo(q, K, V, first, scale, group):
    n, Hq, D = q.shape
    Hkv = K.shape[1]
    out = np.empty((n, Hq, D))
    for h in range(Hq):
        out[:, h:h + 1] = _real(q[:, h:h + 1], K[:, h % Hkv:h % Hkv + 1],
                                V[:, h % Hkv:h % Hkv + 1], first, scale, 1)
    return out


def _mut_kv_swap(q, K, V, first, scale, group):
    return _real(q, V, K, first, scale, group)


def _mut_exclusive_window(q, K, V, first, scale, group):
    # attends keys 0..p-1 instead of 0..p (the query's own key left out)
    n = q.shape[0]
    out = _real(q, K, V, first, scale, group)
    for i in range(n):
        p = first + i
        if p >= 1:
            out[i:i + 1] = _real(q[i:i + 1], K[:p], V[:p], p - 1, scale, group)
    return out


def _check(w):
    kp, vp = _pools(w)
    out = _attn(w, kp, vp)
    causal = bool(np.all(w.query_lens == w.context_lens))
    for s in range(w.num_seqs):
        t0, t1 = w.query_start_loc[s], w.query_start_loc[s + 1]
        ref = _sdpa_seq(w, kp, vp, s, causal=causal)
        if not np.allclose(out[t0:t1], ref, rtol=0, atol=1e-10):
            return False
    return True


def _cases():
    return [make_workload([10, 40, 33], [1, 1, 1], num_q_heads=8, num_kv_heads=2, head_dim=16,
                          seed=31),
            make_workload([37, 9], [37, 9], num_q_heads=4, num_kv_heads=2, head_dim=16,
                          seed=32)]


def test_real_oracle_passes():
    assert all(_check(w) for w in _cases())


@pytest.mark.parametrize("mutant", [_mut_no_scale, _mut_gqa_modulo, _mut_kv_swap,
                                    _mut_exclusive_window])
def test_mutant_is_caught(monkeypatch, mutant):
    monkeypatch.setattr(pa, "_attend", mutant)
    assert not all(_check(w) for w in _cases())
