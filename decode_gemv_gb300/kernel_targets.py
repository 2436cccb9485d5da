"""Run one library call on a full-size workload matrix a few times, for
profiler captures of a single kernel (e.g. ``ncu -k regex:q_lut -s 2 -c 1``):

    python -m decode_gemv_gb300.kernel_targets <target> [--reps N]

Targets (matrices from the seeded workload generators, encoded on the host,
uploaded once; every call on the same device buffers):

  gate_q4            lw_decode_gemv, Mistral-7B-shaped gate 14336x4096, 4-bit coded
  gate_q4_twin       lw_twin_gemv on the same matrix's fixed-width twin
  gate_q4_b16        lw_decode_gemm, batch 16 (tensor-core route)
  gate_q4_b32        lw_decode_gemm, batch 32
  gate_q4_decode     lw_decode (decode only) of the 4-bit gate
  llama_gate_bf16    lw_decode_gemv, Llama-3.1-8B MLP gate, BF16 exponent coding
  llama_gate_bf16_b16      lw_decode_gemm of the same, batch 16 (tensor cores)
  llama_gate_bf16_b64      lw_decode_gemm of the same, batch 64 (tensor cores)
  llama_gate_bf16_decode   lw_decode of the same

Exits nonzero if a call reports a device status."""
import argparse
import sys

import torch

from decode_gemv_gb300 import inputs, lw

TARGETS = ("gate_q4", "gate_q4_twin", "gate_q4_b16", "gate_q4_b32", "gate_q4_decode",
           "llama_gate_bf16", "llama_gate_bf16_b16", "llama_gate_bf16_b64", "llama_gate_bf16_decode")


def main(argv=None) -> int:
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("target", choices=TARGETS)
    p.add_argument("--reps", type=int, default=3)
    args = p.parse_args(argv)
    lw.load()
    dev = "cuda"
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    t = args.target
    if t.startswith("gate_q4"):
        spec = inputs.workload_specs(inputs.MISTRAL_LAYER)[4]
        batch = 16 if t.endswith("b16") else 32 if t.endswith("b32") else 1
        m = inputs.make_matrix(inputs.MISTRAL_LAYER, spec, 0, 4, batch=batch)
        hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"],
                                 twin=t.endswith("twin"))
        X = torch.from_numpy(m["x"]).to(dev)
    else:
        spec = inputs.workload_specs(inputs.LLAMA_MLP_BF16)[0]
        batch = 16 if t.endswith("b16") else 64 if t.endswith("b64") else 1
        m = inputs.make_matrix(inputs.LLAMA_MLP_BF16, spec, 0, 0, batch=batch)
        hb = lw.lw_encode_bundle(lw.LW_FMT_BF16_EXP, m["bits"], None, None)
        X = torch.from_numpy(m["x"].view("int16")).to(dev).reshape(batch, -1)
    db = lw.DeviceBundle.upload(hb, dev)
    if t.endswith("decode"):
        if db.fmt == lw.LW_FMT_Q4_PAIR:
            out = torch.zeros(spec.rows * spec.cols // 2, dtype=torch.uint8, device=dev)
        else:
            out = torch.zeros(spec.rows * spec.cols, dtype=torch.int16, device=dev)
        for _ in range(args.reps):
            lw.lw_decode(db, out, st)
    else:
        Y = torch.empty((batch, spec.rows), dtype=torch.float32, device=dev)
        ws = torch.zeros(lw.lw_workspace_bytes(db, batch) // 4 + 64, dtype=torch.float32, device=dev)
        for _ in range(args.reps):
            if t.endswith("twin"):
                lw.lw_twin_gemv(db, X[0], Y[0], ws, st)
            elif batch == 1:
                lw.lw_decode_gemv(db, X[0], Y[0], ws, st)
            else:
                lw.lw_decode_gemm(db, X, batch, Y, ws, st)
    torch.cuda.synchronize()
    code = int(st.item())
    print(f"{t}: {args.reps} calls, device status {code}")
    return 1 if code else 0


if __name__ == "__main__":
    sys.exit(main())
