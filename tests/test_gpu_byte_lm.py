"""The byte-level LM forward on the GPU, stage by stage, against the oracle's
composition and against the frozen identity cards (raw-bit SHA-256 a stage,
tests/golden/identity_cards_v1.json, written from the oracle alone): the
embedding gather, both blocks, the logits, the per-token losses and their
mean, at the byte-LM GEMM shapes (16 x 128 tokens, 64 wide, 4 heads, SwiGLU
172, 256 byte ids)."""
import json
import os

import numpy as np
import pytest

import oracle_models
from bitcmp import assert_bitwise, card
from bitwise_reproducible_fp32_gb300 import byte_lm, inputs
from gpu_util import host, need_gpu, to_dev, torch

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def dev():
    return need_gpu()


def test_byte_lm_forward_stage_cards(dev):
    c = inputs.byte_lm_cfg2()
    cd = dict(c)
    cd["tokens"] = torch.from_numpy(c["tokens"]).cuda()
    cd["labels"] = torch.from_numpy(c["labels"]).cuda()
    cd["emb"], cd["head"] = to_dev(c["emb"]), to_dev(c["head"])
    cd["blocks"] = [{k: to_dev(v) for k, v in b.items()} for b in c["blocks"]]
    got = {k: host(v) for k, v in byte_lm.forward(cd, torch.device("cuda")).items()}
    want = oracle_models.byte_lm_forward(c)
    frozen = json.load(open(os.path.join(GOLDEN, "identity_cards_v1.json")))["cards"]
    assert list(got) == list(want)
    for name in want:
        assert_bitwise(got[name].reshape(want[name].shape), want[name], name)
        assert card(got[name]) == frozen[f"byte_lm/{name}"], name
    assert np.isfinite(got["loss_mean"]).all()


def test_byte_lm_training_step_stage_cards(dev):
    # forward, backward and AdamW: 73 stages, each bit-identical to the oracle's
    # composition and to its frozen card
    c = inputs.byte_lm_cfg2()
    cd = dict(c)
    cd["tokens"] = torch.from_numpy(c["tokens"]).cuda()
    cd["labels"] = torch.from_numpy(c["labels"]).cuda()
    cd["emb"], cd["head"] = to_dev(c["emb"]), to_dev(c["head"])
    cd["blocks"] = [{k: to_dev(v) for k, v in b.items()} for b in c["blocks"]]
    got = {k: host(v) for k, v in
           byte_lm.train_step(cd, torch.device("cuda"), inputs.BYTE_LM_HP).items()}
    want = oracle_models.byte_lm_step(c, inputs.BYTE_LM_HP)
    frozen = json.load(open(os.path.join(GOLDEN, "identity_cards_v1.json")))["cards"]
    assert list(got) == list(want)
    for name in want:
        assert_bitwise(got[name].reshape(want[name].shape), want[name], name)
        assert card(got[name]) == frozen[f"byte_lm_step/{name}"], name


def test_byte_lm_training_step_replayed_from_a_cuda_graph(dev):
    # the step captured once (its 120 launches) and replayed: the same 73
    # stage cards as the eager step
    c = inputs.byte_lm_cfg2()
    cd = dict(c)
    cd["tokens"] = torch.from_numpy(c["tokens"]).cuda()
    cd["labels"] = torch.from_numpy(c["labels"]).cuda()
    cd["emb"], cd["head"] = to_dev(c["emb"]), to_dev(c["head"])
    cd["blocks"] = [{k: to_dev(v) for k, v in b.items()} for b in c["blocks"]]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    device = torch.device("cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # warm-up off the capture
        byte_lm.train_step(cd, device, inputs.BYTE_LM_HP, status=status)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = byte_lm.train_step(cd, device, inputs.BYTE_LM_HP, status=status)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    frozen = json.load(open(os.path.join(GOLDEN, "identity_cards_v1.json")))["cards"]
    for name, t in st.items():
        assert card(host(t)) == frozen[f"byte_lm_step/{name}"], name
