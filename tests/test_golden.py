"""The oracle against its stored regression fixture (CPU only)."""
import json
import os

import numpy as np

from golden.make_golden import OUT, compute


def test_oracle_matches_stored_fixture():
    stored = json.load(open(OUT))["values"]
    now = compute()
    assert stored.keys() == now.keys()
    for k in stored:
        a, b = np.array(now[k]), np.array(stored[k])
        assert a.shape == b.shape, k
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13, err_msg=k)
