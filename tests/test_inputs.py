"""The synthetic 162M decoder has the model card's parameter count ("MojoLearn
162M" model card, table "Compared with GPT-3 Small": 162,147,840 parameters,
12 layers, 768 wide, SwiGLU 2,048, untied 50,257-id embeddings), and its
token ids and labels are the next-token pairs of one draw."""
import numpy as np

from bitwise_reproducible_fp32_gb300 import inputs


def test_decoder_162m_parameter_count_and_shapes():
    c = inputs.decoder_162m()
    n = c["emb"].size + c["head"].size + sum(v.size for b in c["blocks"] for v in b.values())
    assert n == 162_147_840
    assert len(c["blocks"]) == 12 and c["heads"] == 12 and c["d"] == 768
    assert c["tokens"].shape == c["labels"].shape == (4 * 2048,)
    assert c["tokens"].min() >= 0 and c["tokens"].max() < 50257
    t = c["tokens"].reshape(4, 2048)
    y = c["labels"].reshape(4, 2048)
    assert np.array_equal(t[:, 1:], y[:, :-1])      # labels are the next tokens
