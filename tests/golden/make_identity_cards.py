"""Writes identity_cards_v1.json: SHA-256 of the oracle's raw output bits on
small seeded workloads of the five configurations (reduced shapes where the
full one is large). It calls only the oracle and the seeded input generators.

The cards freeze profile v1: a change in any oracle arithmetic changes a card,
and a deliberate change must come with a new profile version, as the
"mojolearn" PyPI page (section "Stability and release cadence") requires of any
numerical change that is not bit-inert.

Run from the repository root: python tests/golden/make_identity_cards.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(HERE))

import oracle                                   # noqa: E402
from bitcmp import card                         # noqa: E402
from bitwise_reproducible_fp32_gb300 import inputs   # noqa: E402


def cards():
    out = {}
    for p in inputs.gemm_cfg1():
        out[f"cfg1/{p['name']}"] = card(oracle.gemm(p["A"], p["B"], p["transA"], p["transB"]))
    for p in inputs.gemm_cfg2():
        out[f"cfg2/{p['name']}"] = card(oracle.gemm(p["A"], p["B"], p["transA"], p["transB"]))
    for p in inputs.gemm_cfg3(tokens=64, d=96, dff=128, vocab=1000):
        out[f"cfg3_small/{p['name']}"] = card(oracle.gemm(p["A"], p["B"], p["transA"], p["transB"]))
    r = inputs.rowops_cfg4(rows=32, d=768, vocab=5003)
    y, inv = oracle.rmsnorm(r["x"], r["gain"], eps=r["eps"])
    out["cfg4_small/rmsnorm_y"] = card(y)
    out["cfg4_small/rmsnorm_inv_rms"] = card(inv)
    loss, d, bad = oracle.xent(r["logits"], r["labels"], with_dlogits=True)
    assert bad == 0
    out["cfg4_small/xent_loss"] = card(loss)
    out["cfg4_small/xent_dlogits"] = card(d)
    out["cfg4_small/xent_loss_mean"] = card(oracle.mean(loss))
    for p in inputs.dw_cfg5(tokens=600, d=64, dff=96):
        out[f"cfg5_small/{p['name']}"] = card(oracle.gemm(p["A"], p["B"], p["transA"], p["transB"]))
    a = inputs.adamw_cfg5(n=100_003)
    pp, mm, vv = oracle.adamw(a["p"], a["g"], a["m"], a["v"], a["lr"], a["beta1"],
                              a["beta2"], a["eps"], a["weight_decay"], a["step"])
    out["cfg5_small/adamw_p"] = card(pp)
    out["cfg5_small/adamw_m"] = card(mm)
    out["cfg5_small/adamw_v"] = card(vv)
    # the byte-level LM forward at the byte-LM GEMM shapes, stage by stage
    import oracle_models
    for name, v in oracle_models.byte_lm_forward(inputs.byte_lm_cfg2()).items():
        out[f"byte_lm/{name}"] = card(v)
    # one whole training step of it (forward, backward, AdamW from zero moments)
    for name, v in oracle_models.byte_lm_step(inputs.byte_lm_cfg2(), inputs.BYTE_LM_HP).items():
        out[f"byte_lm_step/{name}"] = card(v)
    return out


if __name__ == "__main__":
    doc = {"profile_version": 1,
           "_generator": "tests/golden/make_identity_cards.py (oracle only)",
           "cards": cards()}
    with open(os.path.join(HERE, "identity_cards_v1.json"), "w") as f:
        json.dump(doc, f, indent=1, sort_keys=True)
        f.write("\n")
    print(f"wrote {len(doc['cards'])} cards")
