"""Child process of the cross-process determinism test (test code only): runs every
entry point of the library once on seeded inputs and prints one JSON object mapping
each entry point to the SHA-256 of its output bytes."""
from __future__ import annotations

import hashlib
import json

import numpy as np
import torch


def _h(*ts):
    m = hashlib.sha256()
    for t in ts:
        m.update(t.detach().contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return m.hexdigest()


def main():
    from weight_only_bit_mlx_gb300 import qlinear as q
    from weight_only_bit_mlx_gb300 import synth

    torch.cuda.set_device(0)
    out = {}
    for bits in (4, 6, 8):
        w = q.QWeight.from_numpy(synth.make_weight(768, 2048, bits, config_id=140, tensor_id=bits))
        w3 = q.QWeight.from_numpy(synth.make_weight(768, 2048, bits, config_id=140, tensor_id=10 + bits))
        x = q.bf16_from_bits(synth.make_x(16, 2048, config_id=140))
        X = q.bf16_from_bits(synth.make_x(300, 2048, config_id=141))
        out[f"qlinear_mv/{bits}"] = _h(q.qlinear_mv(w, x[3]))
        out[f"qlinear_mv_rows/{bits}"] = _h(q.qlinear_mv_rows(w, x))
        out[f"qffn_swiglu_mv/{bits}"] = _h(q.qffn_swiglu_mv(w, w3, x))
        out[f"qattn_proj_mv/{bits}"] = _h(*q.qattn_proj_mv(w, w3, w, w3, x[:5]))
        out[f"qlinear_pgemm/{bits}"] = _h(q.qlinear_pgemm(w, X))
        Y = torch.empty(300, 768, device="cuda")
        out[f"qlinear_pgemm_noalloc/{bits}"] = _h(q.qlinear_pgemm_noalloc(w, X, Y))
        A = q.qlinear_pgemm(w3, X)
        out[f"qlinear_pgemm_swiglu/{bits}"] = _h(q.qlinear_pgemm_swiglu(w, X, A))
        rp = q.bf16_from_bits(synth.make_bf16((300, 768), config_id=142, tensor_id=1))
        gp = q.bf16_from_bits(synth.make_bf16((768,), 0.5, 1.5, config_id=143, tensor_id=1))
        out[f"qlinear_pgemm_resid_norm/{bits}"] = _h(q.qlinear_pgemm_resid_norm(w, X, rp, gp, 1e-5), rp)
        r = q.bf16_from_bits(synth.make_bf16((16, 768), config_id=142))
        g = q.bf16_from_bits(synth.make_bf16((768,), 0.5, 1.5, config_id=143))
        o = q.qlinear_mv_resid_norm(w, x, r, g, 1e-5)
        out[f"qlinear_mv_resid_norm/{bits}"] = _h(o, r)
    a = torch.from_numpy(synth.make_f32(4, 1024, 2.0, config_id=144)).cuda()
    c = torch.from_numpy(synth.make_f32(4, 1024, 1.0, config_id=145)).cuda()
    out["qswiglu"] = _h(q.qswiglu(a, c))
    hd, nq, nkv, ring = 64, 8, 2, 16
    qf = torch.from_numpy(synth.make_f32(3, nq * hd, 2.0, config_id=146, tensor_id=1)).cuda()
    kf = torch.from_numpy(synth.make_f32(3, nkv * hd, 2.0, config_id=146, tensor_id=2)).cuda()
    vf = torch.from_numpy(synth.make_f32(3, nkv * hd, 1.0, config_id=146, tensor_id=3)).cuda()
    nw = q.bf16_from_bits(synth.make_bf16((hd,), 0.5, 1.5, config_id=146, tensor_id=4))
    pos = torch.tensor([0, 77, 1 << 20], dtype=torch.int32, device="cuda")
    kr = torch.zeros(3, ring, nkv * hd, dtype=torch.bfloat16, device="cuda")
    vr = torch.zeros_like(kr)
    qo = q.qattn_qknorm_rope_kv(qf, kf, vf, nq, nkv, hd, 32, 1e6, 1e-5, nw, nw, pos, kr, vr)
    out["qattn_qknorm_rope_kv"] = _h(qo, kr, vr)
    y = torch.from_numpy(synth.make_f32(3, 1024, 0.5, config_id=147)).cuda()
    r = q.bf16_from_bits(synth.make_bf16((3, 1024), config_id=148))
    g = q.bf16_from_bits(synth.make_bf16((1024,), 0.5, 1.5, config_id=149))
    out["qresid_rmsnorm"] = _h(q.qresid_rmsnorm(y, r, g, 1e-5), r)
    torch.cuda.synchronize()
    out["status"] = q.qlinear_last_error()
    print(json.dumps(out, sort_keys=True))


if __name__ == "__main__":
    main()
