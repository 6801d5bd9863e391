"""The seeded input generators: determinism, recipe facts and bit-exact casts."""
import json
import os

import numpy as np
import torch

import synth


def test_prefill_is_deterministic_and_shaped():
    a = synth.prefill(synth.C1)
    b = synth.prefill(synth.C1)
    for t in ("q", "k", "v"):
        assert a[t].shape == (1, 2, 512, 64) and a[t].dtype == np.uint16
        assert (a[t] == b[t]).all()
    assert not (a["q"] == a["k"]).all()


def test_diffuse_fraction_is_exactly_a_quarter():
    cfg = synth.C2.replace(s=1024, hq=2, hk=2)
    x = synth.bits_to_f64(synth.prefill(cfg)["k"], "bf16")
    for h in range(2):
        blocks = x[0, h].reshape(-1, 64, cfg.d)
        spread = blocks.std(axis=1).mean(axis=1)  # ~0.3 or ~1.5 per block
        assert (spread > 0.9).sum() == 4 and (spread < 0.6).sum() == 12


def test_bf16_and_f16_casts_match_torch():
    x = np.random.default_rng(3).standard_normal(100000).astype(np.float32) * 7
    tb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (synth.f32_to_bf16_bits(x) == tb).all()
    th = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert (synth.f32_to_f16_bits(x) == th).all()
    assert (synth.bits_to_f64(tb, "bf16") ==
            torch.from_numpy(x).to(torch.bfloat16).double().numpy()).all()


def test_cache_rows_numpy_and_torch_agree():
    cfg = synth.C5
    rows = np.arange(1000, 1400)
    a = synth.cache_rows(cfg, rows)
    b = synth.cache_rows_torch(cfg, 1000, 1400, "cpu").view(torch.int16).numpy().view(np.uint16)
    assert (a == b).all()
    v = synth.bits_to_f64(a, "bf16")
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01


def test_decode_inputs():
    cfg = synth.C5.replace(n_queries=8)
    x = synth.decode(cfg)
    assert x["q"].shape == (8, 16, 576)
    assert sorted(x["page_table"].ravel().tolist()) == list(range(cfg.n_pages))
    for c in range(8):
        row = x["idx"][c]
        assert row.shape == (2048,) and (np.diff(row) > 0).all()
        assert row[0] >= 0 and row[-1] < cfg.tokens_per_query


def test_decode_scale_matches_its_calibration_record():
    path = os.path.join(os.path.dirname(__file__), "golden", "decode_sm_scale.json")
    rec = json.load(open(path))
    assert rec["seed"] == synth.C5.seed
    assert rec["sm_scale"] == synth.C5.sm_scale
    assert abs(rec["median_n_eff"] - 15.0) < 0.5


def test_sample_qblocks_holds_first_and_last():
    units = synth.sample_qblocks(synth.C3, 8)
    per = {}
    for b, h, i in units:
        per.setdefault((b, h), []).append(i)
    assert len(per) == 64
    for v in per.values():
        assert 0 in v and 255 in v and len(v) == 8
