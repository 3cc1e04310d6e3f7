"""DiT decision records from host copies of the mode words and policy states (CPU only).

A record carries the mode and flags of the word and the policy values held in
the block's state after the decision. Γ is absent before the first computed
step and the cosine before the second. Non-finite values are written as
strings, so a record stays strict JSON.
"""
import json

import numpy as np


def test_decode_decisions_records():
    from video_dit_mixed_gb300 import abi, dit
    st = [abi.PolicyState() for _ in range(3)]
    st[1].n_computed, st[1].have_gamma, st[1].gamma = 1, 1, 0.04
    st[2].n_computed, st[2].have_gamma, st[2].gamma, st[2].cos, st[2].acc = 3, 1, float("inf"), 0.995, 0.005
    states = np.stack([np.frombuffer(bytes(s), dtype=np.uint8) for s in st])
    assert states.shape == (3, 80)
    modes = np.array([abi.MODE_INT8 | abi.FLAG_POSTSKIP, abi.MODE_NVFP4,
                      abi.MODE_SKIP | abi.FLAG_NEAR], dtype=np.int32)
    r = dit.decode_decisions(modes, states)
    assert r[0] == dict(block=0, mode="INT8", refresh=False, pdr=False, post_skip=True, near=False,
                        gamma=None, cos=None, acc=0.0, n_computed=0)
    assert r[1]["mode"] == "NVFP4" and r[1]["gamma"] == 0.04 and r[1]["cos"] is None
    assert r[2] == dict(block=2, mode="SKIP", refresh=False, pdr=False, post_skip=False, near=True,
                        gamma="inf", cos=0.995, acc=0.005, n_computed=3)
    for rec in r:
        assert json.loads(json.dumps(rec, allow_nan=False)) == rec
    bpr = np.array([abi.MODE_BF16 | abi.FLAG_PDR | abi.FLAG_REFRESH], dtype=np.int32)
    d = dit.decode_decisions(bpr, states[2:])[0]
    assert (d["mode"], d["pdr"], d["refresh"], d["post_skip"]) == ("BF16", True, True, False)
