"""Golden fixtures: the model card's printed shapes and counts, and the frozen
identity cards of the oracle (profile v1)."""
import json
import os
import sys

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))

from bitwise_reproducible_fp32_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_model_card_parameter_count():
    # "MojoLearn 162M" model card, table "Compared with GPT-3 Small": 12 layers
    # of width 768, SwiGLU 2,048 wide (three matrices), no biases, RMSNorm
    # (two gains per block, no final norm), untied input and output tables of
    # 50,257 x 768, and 162,147,840 parameters in all
    card = json.load(open(os.path.join(GOLDEN, "model_card_162m.json")))
    d, f, V, L = card["width"], card["swiglu_width"], card["vocab"], card["layers"]
    per_block = 4 * d * d + 3 * d * f + 2 * d
    assert 2 * V * d + L * per_block == card["parameters"]
    assert inputs.N_PARAMS == card["parameters"]
    assert (inputs.D_MODEL, inputs.D_FF, inputs.VOCAB) == (d, f, V)
    # one shard is 4 sequences of the 2,048-token context: the workloads'
    # 8,192-token batch
    assert inputs.TOKENS == card["shard_sequences"] * card["context"]
    assert card["shards"] * inputs.TOKENS == card["tokens_per_step"]
    hp = inputs.ADAMW_HP
    assert (hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], hp["lr"]) == (
        card["adamw_beta1"], card["adamw_beta2"], card["adamw_eps"],
        card["weight_decay"], card["peak_lr"])


def test_identity_cards_reproduce():
    import make_identity_cards as mk
    want = json.load(open(os.path.join(GOLDEN, "identity_cards_v1.json")))
    assert want["profile_version"] == 1
    got = mk.cards()
    bad = {k: (got.get(k), v) for k, v in want["cards"].items() if got.get(k) != v}
    assert not bad, f"profile v1 identity cards changed: {sorted(bad)}"
