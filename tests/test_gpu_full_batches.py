"""Full-size parity at every (workload, batch) the sweeps report, through the
C ABI, on sampled output rows against the fp64 oracle (tolerance 1e-3,
normwise and componentwise):

* the Mistral-7B-shaped 4-bit q, gate and down at batches 2, 4 and 8 (the
  CUDA-core batched passes, and from 6 rows the tensor-core route);
* the Llama-3.1-8B MLP gate and up (BF16 exponent coding) at batches 16 and
  64 on the tensor-core path;
* one layer of the 32-layer stack variant with a BF16 MLP (4-bit attention
  projections of the stack, BF16 MLP) at batches 2, 8 and 32.

The rows are the same call a user makes (lw_decode_gemm with the whole
batch); each matrix is drawn by the seeded generators the sweeps use."""
import numpy as np
import pytest

import oracle
from decode_gemv_gb300 import inputs
from decode_gemv_gb300 import lw
from helpers import assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lw.load()


FMT = {inputs.Q4: lw.LW_FMT_Q4_PAIR, inputs.Q6: lw.LW_FMT_Q6, inputs.BF16: lw.LW_FMT_BF16_EXP}
ORACLE_FMT = {inputs.Q4: oracle.Q4, inputs.Q6: oracle.Q6, inputs.BF16: oracle.BF16}


def upload(spec, m):
    payload = m["bits"] if spec.fmt == inputs.BF16 else m["codes"]
    hb = lw.lw_encode_bundle(FMT[spec.fmt], payload, m.get("scales"), m.get("mins"))
    return lw.DeviceBundle.upload(hb, DEV)


def product(db, x):
    """lw_decode_gemm (lw_decode_gemv for one row) of the activation rows x."""
    B = x.shape[0]
    X = torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    Y = torch.full((B, db.rows), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(max(1, lw.lw_workspace_bytes(db, B) // 4), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    if B == 1:
        lw.lw_decode_gemv(db, X, Y, ws, st)
    else:
        lw.lw_decode_gemm(db, X, B, Y, ws, st)
    torch.cuda.synchronize()
    return Y.cpu().numpy(), int(st.item())


def sample_rows(n, step):
    return np.unique(np.concatenate([np.arange(0, n, step), [n - 1]]))


def reference(spec, m, rows, x):
    """Oracle outputs and |w||x| row sums of the sampled rows for activations x."""
    sub = {k: v for k, v in m.items() if k not in ("x", "sd")}
    for k in ("codes", "scales", "mins", "bits"):
        if sub.get(k) is not None:
            sub[k] = m[k][rows]
    sub["x"] = x
    f = ORACLE_FMT[spec.fmt]
    return oracle.reference_output(f, sub), oracle.abs_row_products(f, sub)


def check(spec, m, db, batches, step):
    rows = sample_rows(spec.rows, step)
    for b in batches:
        x = m["x"][:b]
        y, st = product(db, x)
        assert st == 0, (spec.name, b, st)
        ref, absprod = reference(spec, m, rows, x)
        assert_close(y[:, rows], ref, absprod)


@pytest.mark.parametrize("index", [0, 4, 6])   # q, gate, down
def test_mistral_q4_small_batches(index):
    spec = inputs.workload_specs(inputs.MISTRAL_LAYER)[index]
    m = inputs.make_matrix(inputs.MISTRAL_LAYER, spec, 0, index, batch=8)
    check(spec, m, upload(spec, m), (2, 4, 8), max(1, spec.rows // 96))


@pytest.mark.parametrize("index", [0, 1])      # gate, up
def test_llama_mlp_bf16_tensor_core(index):
    spec = inputs.workload_specs(inputs.LLAMA_MLP_BF16)[index]
    m = inputs.make_matrix(inputs.LLAMA_MLP_BF16, spec, 0, index, batch=64)
    check(spec, m, upload(spec, m), (16, 64), 131)


def test_llama_mlp_bf16_twin_tensor_core():
    """The direct-palette twin of the full-size gate on the tensor cores at
    batches 16 and 64 (lw_twin_gemm), sampled rows against the oracle."""
    spec = inputs.workload_specs(inputs.LLAMA_MLP_BF16)[0]
    m = inputs.make_matrix(inputs.LLAMA_MLP_BF16, spec, 0, 0, batch=64)
    hb = lw.lw_encode_bundle(lw.LW_FMT_BF16_EXP, m["bits"], twin=True)
    dt = lw.DeviceBundle.upload(hb, DEV)
    rows = sample_rows(spec.rows, 131)
    for b in (16, 64):
        x = m["x"][:b]
        X = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(DEV)
        Y = torch.full((b, spec.rows), float("nan"), dtype=torch.float32, device=DEV)
        ws = torch.zeros(lw.lw_workspace_bytes(dt, b) // 4, dtype=torch.float32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        lw.lw_twin_gemm(dt, X, b, Y, ws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ref, absprod = reference(spec, m, rows, x)
        assert_close(Y.cpu().numpy()[:, rows], ref, absprod)


def stack_bf16mlp_layer(layer):
    """(workload, index, spec) of one layer of the stack with a BF16 MLP: the
    stack's q, k, v, o and the BF16 MLP's gate, up, down."""
    att = inputs.workload_specs(inputs.DECODE_STACK)[:4]
    mlp = inputs.workload_specs(inputs.LLAMA_MLP_BF16)
    return ([(inputs.DECODE_STACK, i, s) for i, s in enumerate(att)]
            + [(inputs.LLAMA_MLP_BF16, i, s) for i, s in enumerate(mlp)])


@pytest.mark.parametrize("which", range(7))
def test_stack_bf16mlp_layer_batches(which):
    workload, index, spec = stack_bf16mlp_layer(0)[which]
    m = inputs.make_matrix(workload, spec, 0, index, batch=32)
    check(spec, m, upload(spec, m), (2, 8, 32), max(1, spec.rows // 64))
