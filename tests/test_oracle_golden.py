"""The oracle against its stored decode of the tiny configuration
(tests/golden/tiny_decode.json, written by tests/golden/make_oracle_golden.py
from the oracle alone): a regression pin — any change of the oracle's
arithmetic shows here and must regenerate the file with its reason."""
import importlib.util
import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def _maker():
    spec = importlib.util.spec_from_file_location("make_oracle_golden",
                                                  os.path.join(HERE, "golden", "make_oracle_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_tiny_decode_matches_the_stored_oracle_run():
    with open(os.path.join(HERE, "golden", "tiny_decode.json")) as fh:
        want = json.load(fh)
    got = _maker().tiny_decode()
    assert got["tokens"] == want["tokens"]
    # float64 through BLAS: the summation order may differ between machines
    np.testing.assert_allclose(got["top2_margin"], want["top2_margin"], rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(got["last_residual_norm"], want["last_residual_norm"], rtol=1e-9)
