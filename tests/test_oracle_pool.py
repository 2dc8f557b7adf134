"""Host logic of the per-head oracle pool used by the full-size GPU parity tests."""
import numpy as np
import torch

from oracle import kda_oracle as O
from kda_delta_rule_gb300 import inputs as I


def test_per_head_pool_matches_the_whole_call():
    """The spawn pool that the full-size GPU parity tests use splits the oracle's prefill by
    head; every head's outputs, final state and checkpoints equal the single whole-array call."""
    from oracle_pool import prefill_chunked_per_head
    S0, p, cu = I.prefill_inputs([200, 130], 3, 16, 8, dtype=torch.float32, seed=21)
    arrs = [S0.numpy()] + [p[n].numpy() for n in ("q", "k", "v", "g", "beta")]
    o, S, ck = O.prefill_chunked(*arrs, cu_seqlens=cu, chunk=64, ckpt_stride=64)
    per = prefill_chunked_per_head(*arrs, cu, 64, range(3))
    for h in range(3):
        oh, Sh, ckh = per[h]
        assert np.array_equal(oh[:, 0], o[:, h]) and np.array_equal(Sh[:, 0], S[:, h])
        assert [(n, t) for n, t, _ in ckh] == [(n, t) for n, t, _ in ck]
        assert all(np.array_equal(a[2][0], b[2][h]) for a, b in zip(ckh, ck))
