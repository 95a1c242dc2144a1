"""Pin of the oracle's dynamic loss-scale rule against torch's own AMP scale update."""
import numpy as np
import torch

import oracle


def test_scaler_matches_torch_amp_update_scale():
    rng = np.random.default_rng(30)
    for growth, backoff, interval in [(2.0, 0.5, 2), (2.0, 0.5, 5), (1.5, 0.25, 3), (2.0, 0.5, 1)]:
        scale, good = 65536.0, 0
        ts = torch.tensor([65536.0])
        tg = torch.tensor([0], dtype=torch.int32)
        for _ in range(200):
            inf = bool(rng.random() < 0.15)
            scale, good = oracle.scaler_update(scale, good, inf, growth, backoff, interval)
            torch._amp_update_scale_(ts, tg, torch.tensor([1.0 if inf else 0.0]), growth,
                                     backoff, interval)
            assert scale == ts.item() and good == tg.item()


def test_scaler_does_not_grow_to_infinity():
    scale, good = 2.0**127, 0
    scale, good = oracle.scaler_update(scale, good, False, 2.0, 0.5, 1)
    assert scale == 2.0**127 and good == 0
