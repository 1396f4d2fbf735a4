"""The per-query-head process pool of the full-length parity tests gives the oracle's
own one-KV-head result (dK/dV summed over the query heads), on a small tree."""
import numpy as np

import workloads as W
from oracle import attention as A
from tests.oracle_pool import oracle_one_kv_head


def test_pool_equals_oracle_on_one_kv_head():
    w = W.custom(W.Tree([40, 7], [[9, 1, 30], [12]]), hq=3, hkv=1, d=16, dtype="fp32", seed=9)
    host = {n: W.tensor_rows_np(w, n) for n in W.TENSORS}
    ref = A.tree_attention_direct(host, w.tree.offsets(), A.default_scale(w.d))
    got = oracle_one_kv_head(host, w.tree.offsets(), A.default_scale(w.d), processes=2)
    for k, v in ref.items():
        np.testing.assert_allclose(got[k], v, rtol=0, atol=1e-12, err_msg=k)
