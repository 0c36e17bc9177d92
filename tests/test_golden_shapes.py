"""The pages' stated split shapes (tests/golden/split_shapes.json) against the
oracle's split/concat helpers."""
import json
import os

import numpy as np
import pytest

from oracle import tp_oracle as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "split_shapes.json")))


@pytest.mark.parametrize("case", GOLD["cases"], ids=[c["id"] for c in GOLD["cases"]])
def test_split_shape_facts(case):
    r = np.random.default_rng(0)
    if case["kind"] == "heads":
        H, n, d, h = case["H"], case["N"], 2, 3
        Wq, Wk, Wv = (r.standard_normal((h, H * d)) for _ in range(3))
        if case["valid"]:
            W = O.pack_qkv(Wq, Wk, Wv, n, d)
            assert W.shape == (n, h, 3, case["expect_per_shard"], d)
        else:
            with pytest.raises(ValueError):
                O.pack_qkv(Wq, Wk, Wv, n, d)
    elif case["kind"] == "columns":
        W = r.standard_normal((3, case["cols"]))
        Ws = O.split_columns_like(W, case["N"])
        assert Ws.shape == (case["N"], 3, case["expect_per_shard"])
        assert np.array_equal(O.concat_columns(Ws), W)
    elif case["kind"] == "column_block":
        W = r.standard_normal((case["M"], case["Ncols"]))
        assert O.split_columns_like(W, case["n"]).shape[1:] == tuple(case["expect_block"])
    elif case["kind"] == "row_block":
        W = r.standard_normal((case["M"], case["Ncols"]))
        X = r.standard_normal((case["B"], case["M"]))
        assert O.split_rows_like(W, case["m"]).shape[1:] == tuple(case["expect_block"])
        assert O.split_columns_like(X, case["m"]).shape[1:] == tuple(case["expect_x_block"])
