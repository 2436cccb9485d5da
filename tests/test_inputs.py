"""The seeded synthetic inputs against the workloads' stated recipes: shapes,
value ranges, distributions, the BF16 outlier rule and determinism.  CPU
only; the generators hold none of the method's arithmetic."""
import numpy as np

from decode_gemv_gb300 import inputs


def _f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def test_workload_shapes():
    shapes = lambda w: [(s.name, s.rows, s.cols) for s in inputs.workload_specs(w)]
    assert shapes(inputs.TINY) == [(shapes(inputs.TINY)[0][0], 256, 1024)]
    assert shapes(inputs.MISTRAL_LAYER) == [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096),
                                            ("o", 4096, 4096), ("gate", 14336, 4096),
                                            ("up", 14336, 4096), ("down", 4096, 14336)]
    assert shapes(inputs.PHI3_LAYER) == [("qkv", 9216, 3072), ("o", 3072, 3072),
                                         ("gate_up", 16384, 3072), ("down", 3072, 8192)]
    assert shapes(inputs.LLAMA_MLP_BF16) == [("gate", 14336, 4096), ("up", 14336, 4096),
                                             ("down", 4096, 14336)]
    assert shapes(inputs.DECODE_STACK) == shapes(inputs.MISTRAL_LAYER)
    # one layer of the Mistral shape: 218,103,808 weights
    assert sum(r * c for _, r, c in shapes(inputs.MISTRAL_LAYER)) == 218_103_808


def test_generation_is_seeded():
    spec = inputs.workload_specs(inputs.MISTRAL_LAYER)[1]
    a = inputs.make_matrix(inputs.MISTRAL_LAYER, spec, 3, 1)
    b = inputs.make_matrix(inputs.MISTRAL_LAYER, spec, 3, 1)
    c = inputs.make_matrix(inputs.MISTRAL_LAYER, spec, 4, 1)
    assert all(np.array_equal(a[k], b[k]) for k in ("codes", "scales", "mins", "x"))
    assert not np.array_equal(a["codes"], c["codes"])
    # the tiny matrix: seed 0, code sd 1.6
    t = inputs.make_matrix(inputs.TINY, inputs.workload_specs(inputs.TINY)[0])
    r = np.random.default_rng(0)
    want = np.clip(np.rint(r.normal(7.5, 1.6, size=(256, 1024))), 0, 15)
    assert np.array_equal(t["codes"], want.astype(np.uint8))


def test_q4_recipe():
    m = inputs.small_q4(11, 512, 4096, sd=1.6)
    c = m["codes"].astype(np.float64)
    assert m["codes"].dtype == np.uint8 and c.min() >= 0 and c.max() <= 15
    assert abs(c.mean() - 7.5) < 0.02
    # rounding adds a uniform error of variance 1/12
    assert abs(c.std() - np.sqrt(1.6 ** 2 + 1 / 12)) < 0.02
    s, mn = _f16(m["scales"]), _f16(m["mins"])
    assert m["scales"].shape == (512, 16) and m["mins"].shape == (512, 16)
    assert s.min() >= 0.005 * (1 - 2 ** -10) and s.max() <= 0.02 * (1 + 2 ** -10)
    assert mn.min() >= -0.1 * (1 + 2 ** -10) and mn.max() <= 0.0
    assert abs(s.mean() - 0.0125) < 0.0005 and abs(mn.mean() + 0.05) < 0.002
    x = m["x"]
    assert x.dtype == np.float32 and x.shape == (1, 4096)
    assert abs(float(x.mean())) < 0.06 and abs(float(x.std()) - 1) < 0.05
    # per-matrix code sd of the layer workloads: U(1.2, 2.2)
    sds = [inputs.make_matrix(inputs.MISTRAL_LAYER, s, 0, i)["sd"]
           for i, s in enumerate(inputs.workload_specs(inputs.MISTRAL_LAYER)[:3])]
    assert all(1.2 <= v <= 2.2 for v in sds) and len(set(sds)) == 3


def test_q6_recipe():
    m = inputs.small_q6(12, 256, 4096)
    c = m["codes"].astype(np.float64)
    assert c.min() >= 0 and c.max() <= 63
    assert abs(c.mean() - 31.5) < 0.03
    assert abs(c.std() - np.sqrt(16 + 1 / 12)) < 0.03
    assert m["scales"].shape == (256, 4096 // 16) and m["mins"] is None
    s = _f16(m["scales"])
    assert s.min() >= 0.005 * (1 - 2 ** -10) and s.max() <= 0.02 * (1 + 2 ** -10)


def test_bf16_recipe():
    p = 0.002
    m = inputs.small_bf16(13, 512, 4096, outlier_p=p)
    bits = m["bits"]
    w = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    base = inputs.small_bf16(13, 512, 4096, outlier_p=0.0)["bits"]
    wb = (base.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(wb.std() - 0.02) < 0.0003 and abs(wb.mean()) < 0.0003
    # outliers: the same draw with the exponent raised by k in 8..20 (an
    # exact multiplication by 2^k), sign and mantissa kept
    diff = bits != base
    rate = diff.mean()
    assert abs(rate - p) < 0.0003
    e, eb = (bits >> 7) & 0xFF, (base >> 7) & 0xFF
    k = e[diff].astype(int) - eb[diff].astype(int)
    assert k.min() >= 8 and k.max() <= 20 and len(np.unique(k)) == 13
    assert np.array_equal(bits[diff] & 0x807F, base[diff] & 0x807F)
    assert np.array_equal(w[diff], wb[diff] * np.exp2(k))
    # activations: bf16 bits of N(0, 1)
    x = (m["x"].astype(np.uint32) << 16).view(np.float32)
    assert m["x"].dtype == np.uint16 and abs(float(x.std()) - 1) < 0.05
