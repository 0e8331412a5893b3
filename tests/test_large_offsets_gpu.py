"""Byte offsets past 2^32 in the stored-dS workspace (GPU).

The deterministic D_qk 128 route stores every visited dS^T tile; on a causal
B1 Hq16 Hkv4 S17408 problem that region is 4.7 GiB, so the tiles of the last
query heads lie more than 4 GiB from its start. The main kernel's stores and
the dQ kernel's loads address them with 64-bit tile offsets; a 32-bit product
anywhere on that path would wrap and corrupt the last heads' dQ. The check
runs the full chain and compares sampled rows (tile edges and sequence ends of
the first and last query and KV heads, plus random rows) with the fp64 oracle.
(The pages' own test list scales such checks down to offset arithmetic; this
one runs at the size where it matters.)
"""
import pytest

import workloads
from harness import make_case

pytestmark = pytest.mark.gpu

W = workloads.Workload
BIG = W("ds_ws_over_4gib", 1, 16, 4, 17408, 17408, 128, 128, causal=True, deterministic=True, seed=97)


def test_ds_workspace_offsets_past_4gib():
    import attention_backward_sdpa_gb300 as pkg
    from test_parity_gpu import _sampled_check
    ws = pkg.workspace_size(BIG.B, BIG.Hq, BIG.Hkv, BIG.Sq, BIG.Skv, BIG.Dqk, BIG.Dv, True,
                            causal=True, bottom_right=False, window_left=-1, window_right=-1,
                            padded=False)
    assert ws > (1 << 32)
    _sampled_check(make_case(BIG))
