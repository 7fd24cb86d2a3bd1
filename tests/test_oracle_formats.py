"""Pins of the oracle's cache formats against things other than the oracle:
the pages' closed-form sizes, library definitions of the FP8/E8M0 formats
(torch), an independent binade-wise formulation of FP4 rounding, and
constructed round trips whose expected bytes are written out here."""
import json
import math
import os

import numpy as np
import pytest
import torch

from gen import inputs as G

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "sizes.json")))


# ------------------------------------------------------------ closed forms
def test_entry_sizes_match_pages(oracle_lib):
    sz = oracle_lib.entry_bytes()
    assert sz["kv"] == GOLD["kv_entry_bytes"] == GOLD["kv_fp4_values"] // 2 + GOLD["kv_fp4_values"] // GOLD["kv_scale_every"]
    assert sz["idx"] == GOLD["idx_key_bytes"] == GOLD["idx_fp4_values"] // 2 + GOLD["idx_fp4_values"] // GOLD["idx_scale_every"]
    assert sz["swa"] == GOLD["swa_entry_bytes"]
    # 2.5 entries per token x (288 + 68) = 890 B/token
    assert GOLD["entries_per_token"] * (sz["kv"] + sz["idx"]) == GOLD["bytes_per_token"]
    # 890 B x 1,048,576 tokens = 0.869140625 GiB, quoted as ~0.87 GiB
    gib = GOLD["bytes_per_token"] * GOLD["context_tokens"] / 2**30
    assert gib == 0.869140625 and round(gib, 2) == GOLD["gib_per_full_sequence_approx"]
    assert GOLD["candidate_positions"] == 2048 * GOLD["pool_block"]


def test_packed_record_lengths(oracle_lib):
    x = G.normal_block_bf16(7, G.S_MISC, 0, 0, 3, 512)
    assert oracle_lib.pack_kv(x).shape == (3, 288)
    assert oracle_lib.pack_swa(x).shape == (3, 528)
    assert oracle_lib.pack_idx(G.normal_block_bf16(7, G.S_MISC, 1, 0, 3, 128)).shape == (3, 68)


# ------------------------------------------------------------ decode tables
def test_e4m3_table_vs_torch(oracle_lib):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle_lib.e4m3_value(b) for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_e8m0_table_vs_torch(oracle_lib):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    got = np.array([oracle_lib.e8m0_value(b) for b in range(256)])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])


OCP_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # OCP Microscaling spec, FP4 E2M1


def test_e2m1_table(oracle_lib):
    for c in range(16):
        v = oracle_lib.e2m1_value(c)
        assert abs(v) == OCP_E2M1[c & 7]
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)


# ------------------------------------------------------------ rounding
def _e2m1_rne_binade(x: float) -> float:
    """Independent formulation: round on each binade's uniform grid with
    numpy's half-to-even rounding, then saturate at 6."""
    a = abs(x)
    if a < 2.0:
        r = np.round(a * 2.0) / 2.0          # grid 0.5 (E2M1 subnormal + first binade)
    elif a < 4.0:
        r = np.round(a)                      # grid 1
    else:
        r = 2.0 * np.round(a / 2.0)          # grid 2
    return math.copysign(min(r, 6.0), x)


def test_e2m1_encode_ties_and_grid(oracle_lib):
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0, 7.0: 6.0, 1e30: 6.0}
    for x, want in ties.items():
        for s in (1.0, -1.0):
            got = oracle_lib.e2m1_value(oracle_lib.e2m1_encode(s * x))
            assert got == s * want, (s * x, got)
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.uniform(-8, 8, 4000), np.arange(-64, 65) / 8.0])
    for x in xs:
        assert oracle_lib.e2m1_value(oracle_lib.e2m1_encode(x)) == _e2m1_rne_binade(x), x


def test_e4m3_encode_vs_torch_in_range(oracle_lib):
    rng = np.random.default_rng(1)
    vals = [oracle_lib.e4m3_value(b) for b in range(127)]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]           # every tie point
    xs = np.concatenate([rng.uniform(-448, 448, 3000), np.exp(rng.uniform(-14, 6, 3000)),
                         np.array(mids), -np.array(mids), np.array(vals)]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_lib.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    # torch keeps the sign of values that round to zero, as the oracle does
    assert np.array_equal(got, ref)


def test_e4m3_saturates(oracle_lib):
    assert oracle_lib.e4m3_encode(1e9) == 0x7E and oracle_lib.e4m3_encode(-500.0) == 0xFE


def test_bf16_from_double_vs_torch(oracle_lib):
    rng = np.random.default_rng(2)
    # doubles that are exact in fp32 so torch's (via-float) path is a single rounding
    xs = rng.standard_normal(3000).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle_lib.bf16_from_double(x) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # a value just above a bf16 tie that fp32 would round onto the tie
    x = 1.0 + 2.0**-8 + 2.0**-40
    assert oracle_lib.bf16_from_double(x) == 0x3F81


# ------------------------------------------------------------ S1 pack
def _bf16(vals):
    return G._f32_to_bf16_bits(np.asarray(vals, np.float32))


def test_pack_kv_roundtrip_every_code_every_scale(oracle_lib):
    """For every finite positive E4M3 scale s and every E2M1 code c, a group
    whose amax is 6*s packs to scale byte s and codes c (expected bytes written
    out from the documented layout: low nibble = even channel, scales at 256+g)."""
    scales = [b for b in range(1, 127)]
    rows, want = [], []
    for si, sb in enumerate(scales):
        s = oracle_lib.e4m3_value(sb)
        x = np.zeros(512, np.float64)
        codes = np.zeros(512, np.int64)
        for g in range(32):
            cs = [(g + i + si) % 16 for i in range(16)]
            cs[(g + si) % 16] = 7                            # amax = 6 s
            for i, c in enumerate(cs):
                x[16 * g + i] = OCP_E2M1[c & 7] * s * (-1 if c & 8 else 1)
                codes[16 * g + i] = c
        xb = _bf16(x)
        assert np.array_equal(G.bf16_bits_to_f32(xb).astype(np.float64), x)  # exact in bf16
        rec = np.zeros(288, np.uint8)
        for c in range(512):
            rec[c // 2] |= (codes[c] << (4 * (c % 2)))
        rec[256:] = sb
        rows.append(xb)
        want.append(rec)
    got = oracle_lib.pack_kv(np.stack(rows))
    assert np.array_equal(got, np.stack(want))


def test_pack_kv_zero_and_underflow_groups(oracle_lib):
    x = np.zeros(512, np.float32)
    x[16:32] = 1e-6           # amax/6 underflows E4M3 -> scale 0, codes 0
    x[32] = -3.0              # ordinary group
    rec = oracle_lib.pack_kv(_bf16(x))[0]
    assert rec[256] == 0 and rec[257] == 0 and np.all(rec[0:16] == 0)
    assert oracle_lib.e4m3_value(rec[258]) == 0.5 and (rec[16] & 15) == 0xF   # -6 * 0.5


def test_pack_kv_matches_library_quantiser(oracle_lib):
    """dequant(pack(x)) == E2M1_binade(x / s) * s with s = torch-E4M3(amax/6)."""
    x = G.normal_block_bf16(11, G.S_MISC, 0, 0, 64, 512)
    xf = G.bf16_bits_to_f32(x).astype(np.float64).reshape(64, 32, 16)
    amax = np.abs(xf).max(axis=2)
    s = torch.from_numpy((amax / 6).astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
    want = np.vectorize(_e2m1_rne_binade)(xf / s[..., None]) * s[..., None]
    got = oracle_lib.dequant_kv(oracle_lib.pack_kv(x)).reshape(64, 32, 16)
    assert np.array_equal(got, want)


# ------------------------------------------------------------ S2 / S3 pack
def _pow2_exp(amax, lim):
    e = math.ceil(math.log2(amax / lim))
    while lim * 2.0**e < amax:
        e += 1
    while lim * 2.0**(e - 1) >= amax:
        e -= 1
    return e


def test_pack_idx_scale_rule_and_values(oracle_lib):
    x = G.normal_block_bf16(12, G.S_MISC, 0, 0, 200, 128)
    rec = oracle_lib.pack_idx(x)
    xf = G.bf16_bits_to_f32(x).astype(np.float64).reshape(200, 4, 32)
    deq = oracle_lib.dequant_idx(rec).reshape(200, 4, 32)
    for r in range(200):
        for g in range(4):
            amax = np.abs(xf[r, g]).max()
            e = int(rec[r, 64 + g]) - 127
            assert e == _pow2_exp(amax, 6.0)                 # smallest 2^e >= amax/6
            want = np.array([_e2m1_rne_binade(v) for v in xf[r, g] / 2.0**e]) * 2.0**e
            assert np.array_equal(deq[r, g], want)


def test_pack_idx_exact_power_of_two_case(oracle_lib):
    x = np.zeros(128, np.float32)
    x[0] = 6.0 * 2.0**-3        # amax/6 = 2^-3 exactly -> scale byte 124, code 7
    x[1] = -0.5 * 2.0**-3
    rec = oracle_lib.pack_idx(_bf16(x))[0]
    assert rec[64] == 124 and rec[0] == (0x9 << 4 | 0x7) and rec[65] == 0   # zero group: byte 0


def test_pack_swa_vs_torch_e4m3(oracle_lib):
    x = G.normal_block_bf16(13, G.S_MISC, 0, 0, 50, 512)
    x[3, :32] = 0                                      # an all-zero group
    rec = oracle_lib.pack_swa(x)
    xf = G.bf16_bits_to_f32(x).astype(np.float64).reshape(50, 16, 32)
    deq = oracle_lib.dequant_swa(rec).reshape(50, 16, 32)
    for r in range(50):
        for g in range(16):
            amax = np.abs(xf[r, g]).max()
            if amax == 0:
                assert rec[r, 512 + g] == 0 and np.all(rec[r, 32 * g:32 * g + 32] == 0)
                continue
            e = _pow2_exp(amax, 448.0)
            assert int(rec[r, 512 + g]) - 127 == e
            q = torch.from_numpy((xf[r, g] / 2.0**e).astype(np.float32)).to(torch.float8_e4m3fn)
            assert np.array_equal(rec[r, 32 * g:32 * g + 32], q.view(torch.uint8).numpy())
            assert np.array_equal(deq[r, g], q.double().numpy() * 2.0**e)


# ------------------------------------------------------------ m=2 pooling
def test_pool_m2_gate_special_cases(oracle_lib):
    x = G.normal_block_bf16(14, G.S_MISC, 0, 0, 8, 512)
    xf = G.bf16_bits_to_f32(x).astype(np.float64)
    z = np.zeros((8, 512), np.float32)
    eq = oracle_lib.pool_m2(x, z)                       # equal logits -> mean
    mean = torch.from_numpy((xf[0::2] + xf[1::2]) / 2).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(eq, mean.astype(np.uint16))
    z[0::2] = 200.0                                     # dominant first logit -> first token
    assert np.array_equal(oracle_lib.pool_m2(x, z), x[0::2])
    z[0::2], z[1::2] = -200.0, 0.0                      # dominant second
    assert np.array_equal(oracle_lib.pool_m2(x, z), x[1::2])


def test_pool_m2_general_within_one_ulp_of_torch_softmax(oracle_lib):
    x = G.normal_block_bf16(15, G.S_MISC, 0, 0, 16, 512)
    z = G.gate_logits_f32(15, 0, np.arange(16), 512)
    got = G.bf16_bits_to_f32(oracle_lib.pool_m2(x, z)).astype(np.float64)
    xf = torch.from_numpy(G.bf16_bits_to_f32(x).astype(np.float64)).view(8, 2, 512)
    p = torch.softmax(torch.from_numpy(z.astype(np.float64)).view(8, 2, 512), dim=1)
    want = (p * xf).sum(1).numpy()
    ulp = np.abs(want) * 2.0**-8 + 1e-40
    assert np.all(np.abs(got - want) <= ulp)
