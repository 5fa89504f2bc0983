"""GPU text generation through the C ABI (``gpt2_sample``): the page
«llm.c：Andrej Karpathy带你从零复现LLM», section «核心代码解读：train_gpt2.c»,
item 5 (sample_mult draws an index from a probability distribution; the
main loop generates a sequence with it).

For every generated position t the test reruns the oracle forward on the
GPU's own tokens and checks that tokens[t] is a valid inverse-CDF draw for
that step's coin under the oracle's probabilities of logits row t-1, with a
tolerance of 1e-5 on the cumulative probabilities (fp32 logits and sums on
the GPU against a float64 prefix sum here).  Where the coin lies farther than
that from every boundary the draw is unique, so the two must agree except at
the rare ties.  Coins come from a seeded generator; expected values from
``oracle/`` only."""
import numpy as np
import pytest

import synth
from oracle import ref

pytestmark = pytest.mark.gpu


def gpu_model(w, **kw):
    import gpt_train_step_02_b300 as g

    return g.GPT2(w, **kw)


def coins_for(n, seed):
    c = np.random.default_rng(seed).random(n).astype(np.float32)
    return np.minimum(c, np.nextafter(np.float32(1.0), np.float32(0.0)))


def check_generation(w, prompt, n_total, seed):
    prompt = np.asarray(prompt, np.int32)
    coins = coins_for(n_total - prompt.size, seed)
    p0 = synth.init_params(w)
    m = gpu_model(w, maxB=1, maxT=n_total)
    m.set_params(p0)
    toks = m.sample(prompt, n_total, coins)
    m.close()
    assert toks.shape == (n_total,)
    np.testing.assert_array_equal(toks[:prompt.size], prompt)
    assert ((toks >= 0) & (toks < w.vocab_size)).all()
    o = ref.RefModel(ref.config_from(w), 1, n_total, np.float32)
    o.set_params(p0)
    agree = 0
    for t in range(prompt.size, n_total):
        o.forward(toks[None, :], None)
        probs = ref.softmax64(o.act("logits").reshape(n_total, -1)[t - 1, :w.vocab_size])
        coin = float(coins[t - prompt.size])
        assert ref.sample_is_valid(probs, coin, int(toks[t]), 1e-5), (t, int(toks[t]), ref.sample_mult(probs, coin))
        agree += int(toks[t] == ref.sample_mult(probs, coin))
    o.close()
    assert agree >= n_total - prompt.size - 1
    return toks


def test_generation_tiny():
    w = synth.WORKLOADS["tiny_L2_C64"]
    check_generation(w, [5, 17, 3], w.max_seq_len, seed=11)


def test_generation_tiny_single_token_prompt_and_determinism():
    w = synth.WORKLOADS["tiny_L2_C64"]
    a = check_generation(w, [0], 20, seed=12)
    b = check_generation(w, [0], 20, seed=12)
    np.testing.assert_array_equal(a, b)


def test_generation_124m_from_end_of_text():
    """The pages' console log starts its generated sequence at id 50256."""
    w = synth.WORKLOADS["gpt2_124m_B4_T64_fp32"]
    check_generation(w, [50256], 12, seed=13)


def test_generation_rejects_bad_arguments():
    import gpt_train_step_02_b300 as g

    w = synth.WORKLOADS["tiny_L2_C64"]
    m = gpu_model(w, maxB=1, maxT=16)
    with pytest.raises(g.GPT2Error):  # a coin of 1 is outside [0, 1)
        m.sample([1], 4, np.array([0.5, 1.0, 0.5], np.float32))
    with pytest.raises(g.GPT2Error):  # longer than the handle's maxT
        m.sample([1], 17, coins_for(16, 1))
    with pytest.raises(g.GPT2Error):  # prompt id outside the vocabulary
        m.sample([w.vocab_size], 4, coins_for(3, 1))
    toks = m.sample([1, 2], 6, coins_for(4, 2))  # the handle still works
    assert toks.shape == (6,)
    m.close()
