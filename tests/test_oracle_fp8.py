"""Pins of the oracle's 8-bit (E4M3) cache and binary16 paths to things other
than themselves.

The pages do not cover an 8-bit KV cache; the format is OCP FP8 E4M3 (OFP8
specification), with a per-tensor scale: stored code = E4M3(x / scale), value
= scale * E4M3 value.  The pins:

* every one of the 256 codes decodes to the value torch's float8_e4m3fn gives
  it (a library implementation of the same format), NaN codes included;
* every one of the 65536 binary16 patterns decodes to torch's float16 value;
* the encoder agrees with torch's float32 -> float8_e4m3fn cast (round to
  nearest even) on every representable value, every midpoint between two
  neighbours (the ties), one float32 step either side of each midpoint, and
  random values at many scales, all within +-448 where torch does not
  saturate; hand-derived codes pin the saturation, NaN, infinities and signed
  zero (tests/golden/e4m3_codes.json);
* the quotient x / scale is the float32 division torch computes;
* attention over an E4M3 cache equals the dense brute force run on the
  torch-decoded values times the scales (no pages, no shared code);
* the quantising append puts each token's codes at the oracle's own slots.

A battery of planted mistakes (compiled from edited copies of the C source)
checks that these pins catch each one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.dense import attention_dense
from support import make_step, to_np64

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _torch_decode(codes):
    return codes.to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _encode_grid():
    """float32 values within +-448 exercising every rounding decision."""
    vals = _torch_decode(torch.arange(256, dtype=torch.int32).to(torch.uint8))
    fin = np.unique(vals[np.isfinite(vals) & (vals >= 0)])
    mids = (fin[:-1] + fin[1:]) / 2  # exact in float32: neighbours differ by one bit
    m32 = mids.astype(np.float32)
    up = np.nextafter(m32, np.float32(np.inf))
    dn = np.nextafter(m32, np.float32(-np.inf))
    g = torch.Generator().manual_seed(77)
    rnd = [(torch.randn(4000, generator=g) * s).numpy() for s in (1e-4, 1e-3, 1e-2, 0.1, 1, 10, 100)]
    x = np.concatenate([fin, mids, up, dn, *rnd]).astype(np.float32)
    x = np.concatenate([x, -x])
    return x[np.abs(x) <= 448]


def _quotient_ties():
    """(x, s) float32 pairs whose float32 quotient x / s is exactly a midpoint
    between two neighbouring E4M3 values (the rounding then depends on the
    quotient being taken in float32)."""
    vals = _torch_decode(torch.arange(256, dtype=torch.int32).to(torch.uint8))
    fin = np.unique(vals[np.isfinite(vals) & (vals > 0)])
    mids = (fin[:-1] + fin[1:]) / 2
    rng = np.random.default_rng(3)
    xs, ss = [], []
    for sc in rng.uniform(0.1, 3.0, 24).astype(np.float32):
        x0 = (mids * np.float64(sc)).astype(np.float32)
        for x in (np.nextafter(x0, np.float32(-np.inf)), x0, np.nextafter(x0, np.float32(np.inf))):
            hit = (x / sc).astype(np.float64) == mids
            xs.append(x[hit])
            ss.append(np.full(hit.sum(), sc, dtype=np.float32))
    x, s = np.concatenate(xs), np.concatenate(ss)
    return np.concatenate([x, -x]), np.concatenate([s, s])


def _fp8_pins_hold(impl) -> bool:
    """The 8-bit pins against ``impl`` (an oracle build); False on any miss."""
    try:
        codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
        if not np.array_equal(oracle.e4m3_decode(codes, impl=impl), _torch_decode(codes),
                              equal_nan=True):
            return False
        x = torch.from_numpy(_encode_grid())
        want = x.to(torch.float8_e4m3fn).view(torch.uint8)
        if not torch.equal(oracle.e4m3_encode(x, impl=impl), want):
            return False
        # a scale: the quotient is torch's float32 division
        xb = (torch.randn(3000, generator=torch.Generator().manual_seed(5)) * 3).to(torch.bfloat16)
        for s in (0.37, 1.7, 1 / 64):
            q = (xb.float() / torch.tensor(s, dtype=torch.float32))
            q = q[q.abs() <= 448]
            ok = (xb.float() / torch.tensor(s, dtype=torch.float32)).abs() <= 448
            if not torch.equal(oracle.e4m3_encode(xb[ok], s, impl=impl),
                               q.to(torch.float8_e4m3fn).view(torch.uint8)):
                return False
        # ties made by the float32 quotient: x / s rounds (in float32) exactly
        # onto a midpoint between two codes while the exact quotient is off it
        xt, st_ = _quotient_ties()
        for sc in np.unique(st_):
            sel = torch.from_numpy(st_ == sc)
            xx = torch.from_numpy(xt)[sel]
            q = xx / torch.tensor(float(sc), dtype=torch.float32)
            if not torch.equal(oracle.e4m3_encode(xx, float(sc), impl=impl),
                               q.to(torch.float8_e4m3fn).view(torch.uint8)):
                return False
        gold = json.load(open(os.path.join(GOLD, "e4m3_codes.json")))["cases"]
        xs = torch.tensor([float(c["x"]) for c in gold], dtype=torch.float32)
        got = oracle.e4m3_encode(xs, impl=impl).tolist()
        if got != [int(c["code"], 16) for c in gold]:
            return False
        # attention over an E4M3 cache vs the dense brute force on decoded values
        for seed, (ks, vs) in enumerate(((0.05, 0.8), (1.0, 1.0), (3.0, 0.02))):
            st = make_step([1, 19, 1, 6], [40, 53, 18, 6], 4, 2, 16, torch.bfloat16, 900 + seed)
            m = st["meta"]
            kc = torch.full(st["oracle_cache"].k.shape, 0x7f, dtype=torch.uint8)
            vc = kc.clone()
            allq = torch.tensor([0] + list(np.cumsum(m.seq_lens_list)), dtype=torch.int32)
            full = oracle.slot_mapping(m.block_table, allq, m.seq_lens, 16, impl=impl)
            kk, vv = torch.cat(st["k_seqs"]), torch.cat(st["v_seqs"])
            oracle.kv_append_e4m3(kc, vc, kk, vv, full, ks, vs, impl=impl)
            # the append stored the encoder's codes at the oracle's slots
            page, off = full // 16, full % 16
            if not torch.equal(kc[page, :, off], oracle.e4m3_encode(kk, ks, impl=impl)):
                return False
            out = oracle.attention(st["q"], kc, vc, m.block_table, m.query_start_loc,
                                   m.seq_lens, 0.3, k_scale=ks, v_scale=vs, impl=impl)
            kd = _torch_decode(oracle.e4m3_encode(kk, ks, impl=impl)) * ks
            vd = _torch_decode(oracle.e4m3_encode(vv, vs, impl=impl)) * vs
            offs = np.cumsum([0] + m.seq_lens_list)
            ref = attention_dense(to_np64(st["q"]), [kd[a:b] for a, b in zip(offs[:-1], offs[1:])],
                                  [vd[a:b] for a, b in zip(offs[:-1], offs[1:])], m.q_lens, 0.3)
            if not np.allclose(out, ref, rtol=0, atol=1e-10):
                return False
        return True
    except (ValueError, AssertionError, IndexError, RuntimeError, TypeError):
        return False


def test_e4m3_pins_hold_for_the_oracle():
    assert _fp8_pins_hold(oracle.lib())


def test_golden_codes_by_hand():
    gold = json.load(open(os.path.join(GOLD, "e4m3_codes.json")))["cases"]
    xs = torch.tensor([float(c["x"]) for c in gold], dtype=torch.float32)
    got = oracle.e4m3_encode(xs)
    for c, g in zip(gold, got.tolist()):
        assert g == int(c["code"], 16), f"{c['x']}: {hex(g)} != {c['code']} ({c['why']})"
    # and back: every finite hand code decodes to its value (saturated ones to 448)
    for c, g in zip(gold, got.tolist()):
        v = float(c["x"])
        if math.isnan(v):
            assert math.isnan(oracle.e4m3_decode(torch.tensor([g], dtype=torch.uint8))[0])


def test_binary16_decoding_matches_torch_on_every_pattern():
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    got = oracle.f16_decode(bits)
    want = bits.view(torch.float16).to(torch.float64).numpy()
    assert np.array_equal(got, want, equal_nan=True)


def test_fp16_queries_and_cache_match_the_dense_brute_force():
    st = make_step([1, 23, 1], [61, 40, 9], 8, 2, 32, torch.float16, 950)
    m = st["meta"]
    oracle.kv_append(st["oracle_cache"].k, st["oracle_cache"].v, st["k_new"], st["v_new"],
                     oracle.slot_mapping(m.block_table, m.query_start_loc, m.seq_lens, 16))
    out = oracle.attention(st["q"], st["oracle_cache"].k, st["oracle_cache"].v, m.block_table,
                           m.query_start_loc, m.seq_lens, 0.2)
    ref = attention_dense(to_np64(st["q"]), [to_np64(x) for x in st["k_seqs"]],
                          [to_np64(x) for x in st["v_seqs"]], m.q_lens, 0.2)
    assert np.allclose(out, ref, rtol=0, atol=1e-10)


FP8_MUTANTS = {
    "e4m3 exponent bias off by one": ("ldexp((double)(8 + m), ef - 10)",
                                      "ldexp((double)(8 + m), ef - 9)"),
    "e4m3 subnormals read as normals": ("double v = ef == 0 ? ldexp((double)m, -9)",
                                        "double v = ef == 0 ? ldexp((double)(8 + m), -10)"),
    "e4m3 NaN code read as a number": ("if (ef == 15 && m == 7) return NAN;", ""),
    "ties rounded away from zero": ("double m = nearbyint(a / ldexp(1.0, e - 3));",
                                    "double m = round(a / ldexp(1.0, e - 3));"),
    "rounding truncates": ("double m = nearbyint(a / ldexp(1.0, e - 3));",
                           "double m = floor(a / ldexp(1.0, e - 3));"),
    "no saturation": ("if (a >= 448.0) return sign | 0x7e;", ""),
    "subnormal spacing wrong": ("int e = -6;", "int e = -7;"),
    "sign dropped": ("uint8_t sign = signbit(y) ? 0x80 : 0x00;", "uint8_t sign = 0x00;"),
    "scale multiplied, not divided": ("float y = xi / scale;", "float y = xi * scale;"),
    "quotient by a reciprocal": ("float y = xi / scale;", "float y = xi * (1.0f / scale);"),
    "k_scale not applied": ("dot *= P->k_scale;", ""),
    "v_scale not applied": ("double pv = p * P->v_scale;", "double pv = p;"),
    "append swaps the scales": ("D, k_scale, k_cache + dst);", "D, v_scale, k_cache + dst);"),
    "binary16 bias off by one": ("ldexp((double)(1024 + fr), ef - 25)", "ldexp((double)(1024 + fr), ef - 24)"),
}


@pytest.mark.parametrize("name", sorted(FP8_MUTANTS))
def test_planted_fp8_mistake_is_caught(name, tmp_path):
    before, after = FP8_MUTANTS[name]
    src = oracle.source_text()
    assert src.count(before) >= 1, f"mutation anchor missing: {before!r}"
    impl = oracle.compile_variant(src.replace(before, after, 1), str(tmp_path / "mutant.so"))
    if name.startswith("binary16"):
        bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
        want = bits.view(torch.float16).to(torch.float64).numpy()
        assert not np.array_equal(oracle.f16_decode(bits, impl=impl), want, equal_nan=True)
    else:
        assert not _fp8_pins_hold(impl), f"pins did not catch: {name}"
