"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times.  Where a full-grid FP64 reference would take too long, the
oracle computes complete rows (or sampled elements) one by one; every other
element is covered by the smaller tests of the same kernels.

Workloads: square uniform 256^3 (four modes); batched 2048 x 64x64x4096 with
padded leading dimensions (tf32, fp16); 8192^3 bf16 with beta = 0.5 and its
unpadded 8191 x 8177 x 8183 tail; 4096^3 log-uniform split vs one-chain vs tf32
vs FFMA; the attention-shaped pair S = Q K^T, O = P V in split mode."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import oracle
import synthetic
from helpers import MODE_Q, TOL, Case, sample_points

pytestmark = pytest.mark.gpu

R, Cm = mpg.ROW_MAJOR, mpg.COL_MAJOR


def row_errors(case, C, rows, q, bi=0):
    sa, sb = case._exps()
    ref, den = oracle.gemm(case.a[bi][rows], case.b[bi], case.c0[bi][rows], case.alpha, case.beta,
                           q, q, sa, sb)
    return oracle.max_rel_err(C[bi][rows], ref, den)


def show(capsys, msg):
    with capsys.disabled():
        print(f"\n[{msg}]")


def test_square_uniform_256_all_modes(capsys):
    mpg.build()
    a = synthetic.uniform((256, 256), synthetic.SEED_A)
    b = synthetic.uniform((256, 256), synthetic.SEED_B)
    errs = {}
    for mode in (mpg.FP16_F32ACC, mpg.BF16_F32ACC, mpg.TF32, mpg.SPLIT_FP16_3CHAIN,
                 mpg.SPLIT_FP16_1CHAIN, mpg.FP32_FFMA):
        c = Case(256, 256, 256, mode, a=a, b=b, alpha=1.0, beta=0.0)
        c.run()
        errs[mode] = c.errors()
    show(capsys, f"square256 (eR, eQ): {errs}")
    assert errs[mpg.FP16_F32ACC][1] <= TOL["q16"]
    assert errs[mpg.BF16_F32ACC][1] <= TOL["q16"]
    assert errs[mpg.TF32][0] <= TOL["tf32"]
    assert errs[mpg.SPLIT_FP16_3CHAIN][0] <= TOL["split"]
    assert errs[mpg.SPLIT_FP16_3CHAIN][0] <= 1.5 * errs[mpg.FP32_FFMA][0]


@pytest.mark.parametrize("mode", [mpg.TF32, mpg.FP16_F32ACC])
def test_batched_2048_padded(mode, capsys):
    mpg.build()
    batch, m, n, k = 2048, 64, 64, 4096
    c = Case(m, n, k, mode, batch=batch, a_layout=R, b_layout=Cm, pad=(8, 8, 8))
    c.run()
    C = c.result()   # also checks that no padding column of any batch was written
    sel = [0, 1, 777, 1024, 2046, 2047]
    eR, eQ = c.errors(C, batches=sel)
    show(capsys, f"batched2048 mode {mode}: eR={eR:.3e} eQ={eQ:.3e}")
    if mode == mpg.TF32:
        assert eR <= TOL["tf32"]
    else:
        assert eQ <= TOL["q16"]


@pytest.mark.parametrize("cta_pair", [0, -1])
def test_large_bf16_8192_beta(cta_pair, capsys):
    """The library's choice (CTA pairs at this size) and single CTAs."""
    mpg.build()
    n = 8192
    c = Case(n, n, n, mpg.BF16_F32ACC, in_dtype="bf16", dist="normal", alpha=1.0, beta=0.5,
             c0=synthetic.normal((n, n), synthetic.SEED_C0), opts=mpg.options(cta_pair=cta_pair))
    c.run()
    C = c.result()
    rows, cols = sample_points(n, n, 3000, 81)
    ref, den = c.reference_points(oracle.Q_NONE, 0, rows, cols)
    err = oracle.max_rel_err(C[0][rows, cols], ref, den)
    err_rows = row_errors(c, C, np.array([0, 4095, 8191]), oracle.Q_NONE)
    show(capsys, f"bf16 8192^3 (cta_pair {cta_pair}): sampled {err:.3e}, rows {err_rows:.3e}")
    assert err <= TOL["q16"] and err_rows <= TOL["q16"]


@pytest.mark.parametrize("ws", ["none", "sizes", "exact"])
def test_large_bf16_tail_unpadded(ws, capsys):
    """8191 x 8177 x 8183 with unpadded leading dimensions: row pitches of
    16366 / 16354 bytes are not multiples of 16, so no TMA descriptor exists:
    without a workspace the generic-load path runs; with the workspace the
    sizes-only query or the exact query asks for, the operands are copied to
    aligned lines and multiplied on the TMA path."""
    import torch
    mpg.build()
    m, n, k = 8191, 8177, 8183
    c = Case(m, n, k, mpg.BF16_F32ACC, in_dtype="bf16", dist="normal", alpha=1.0, beta=0.5,
             c0=synthetic.normal((m, n), synthetic.SEED_C0))
    assert c.lda == k and c.ldb == n and c.ldc == n
    if ws == "none":
        c.run(workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))
    else:
        c.run(exact_ws=(ws == "exact"))
    C = c.result()
    rows, cols = sample_points(m, n, 10000, 82)
    ref, den = c.reference_points(oracle.Q_NONE, 0, rows, cols)
    err = oracle.max_rel_err(C[0][rows, cols], ref, den)
    # whole rows: the first, the last, and rows in the last (ragged) row tile
    err_rows = row_errors(c, C, np.array([0, 1, 4095, 8064, 8127, 8128, 8189, 8190]), oracle.Q_NONE)
    show(capsys, f"bf16 tail (workspace {ws}): sampled {err:.3e}, rows {err_rows:.3e}")
    assert err <= TOL["q16"] and err_rows <= TOL["q16"]


def test_loguniform_4096_split_vs_one_chain_vs_tf32_vs_ffma(capsys):
    mpg.build()
    n = 4096
    a = synthetic.loguniform_signed((n, n), synthetic.SEED_A)
    b = synthetic.loguniform_signed((n, n), synthetic.SEED_B)
    # 69 whole rows: every 64th, and rows at the ends of row tiles
    rows = np.unique(np.concatenate([np.arange(0, 4096, 64), np.array([1, 63, 127, 2047, 4095])]))
    errs = {}
    onload = mpg.options(prepass=-1)
    for mode in (mpg.SPLIT_FP16_3CHAIN, mpg.SPLIT_FP16_1CHAIN, mpg.TF32, mpg.FP32_FFMA):
        c = Case(n, n, n, mode, a=a, b=b, b_layout=Cm, alpha=1.0, beta=0.0, opts=onload)
        c.run()
        C = c.result()
        errs[mode] = row_errors(c, C, rows, oracle.Q_NONE)
        if mode in (mpg.SPLIT_FP16_3CHAIN, mpg.SPLIT_FP16_1CHAIN):
            errs[(mode, "Q")] = row_errors(c, C, rows, MODE_Q[mode])
    # the library's default at this size: the separate conversion pass
    c = Case(n, n, n, mpg.SPLIT_FP16_3CHAIN, a=a, b=b, b_layout=Cm)
    c.run()
    errs["split3 default (conversion pass)"] = row_errors(c, c.result(), rows, oracle.Q_NONE)
    # the three-chain split without chunked accumulation, for the record
    c = Case(n, n, n, mpg.SPLIT_FP16_3CHAIN, a=a, b=b, b_layout=Cm, opts=mpg.options(split_chunk_k=-1))
    c.run()
    errs["split3 one chunk"] = row_errors(c, c.result(), rows, oracle.Q_NONE)
    show(capsys, "loguniform4096 errors vs FP64: " + ", ".join(
        f"{k}: {v:.3e}" for k, v in errs.items()))
    assert errs[mpg.SPLIT_FP16_3CHAIN] <= TOL["split"]
    assert errs[mpg.SPLIT_FP16_3CHAIN] <= 1.5 * errs[mpg.FP32_FFMA]
    assert errs["split3 default (conversion pass)"] <= TOL["split"]
    assert errs[mpg.TF32] <= TOL["tf32"]
    assert errs[(mpg.SPLIT_FP16_3CHAIN, "Q")] <= TOL["q16"]
    assert errs[(mpg.SPLIT_FP16_1CHAIN, "Q")] <= TOL["q16"]


def test_attention_pair_split3(capsys):
    mpg.build()
    q, kk, p, v = synthetic.attention_inputs()
    rows = np.array([0, 1, 1023, 2047])
    # S = Q K^T: B = K^T, i.e. K's row-major storage is B column-major
    cs = Case(2048, 32768, 128, mpg.SPLIT_FP16_3CHAIN, a=q, b=np.ascontiguousarray(kk.T), b_layout=Cm,
              c0=np.zeros((2048, 32768), np.float32))
    cs.run()
    S = cs.result()
    e_s = row_errors(cs, S, rows, oracle.Q_NONE)
    # the same product converted on load (the default above takes the separate pass)
    cl = Case(2048, 32768, 128, mpg.SPLIT_FP16_3CHAIN, a=q, b=np.ascontiguousarray(kk.T), b_layout=Cm,
              c0=np.zeros((2048, 32768), np.float32), opts=mpg.options(prepass=-1))
    cl.run()
    e_sl = row_errors(cl, cl.result(), rows, oracle.Q_NONE)
    # the two-accumulator form (hh; hl + lh), on the pass's copies and on load
    e_sh = []
    for pre in (0, -1):
        ch = Case(2048, 32768, 128, mpg.SPLIT_FP16_3CHAIN, a=q, b=np.ascontiguousarray(kk.T), b_layout=Cm,
                  c0=np.zeros((2048, 32768), np.float32), opts=mpg.options(prepass=pre, split_lo_shared=1))
        ch.run()
        e_sh.append(row_errors(ch, ch.result(), rows, oracle.Q_NONE))
        del ch
    # O = P V; P holds probabilities (<= 1): operand scale 2^14 lifts it out
    # of fp16's subnormal range
    co = Case(2048, 128, 32768, mpg.SPLIT_FP16_3CHAIN, a=p, b=v, c0=np.zeros((2048, 128), np.float32),
              opts=mpg.options(split_exp_a=14))
    co.run()
    O = co.result()
    e_o = row_errors(co, O, np.arange(0, 2048, 64), oracle.Q_NONE)
    # the same product without the operand scale, for the record
    cu = Case(2048, 128, 32768, mpg.SPLIT_FP16_3CHAIN, a=p, b=v, c0=np.zeros((2048, 128), np.float32))
    cu.run()
    e_u = row_errors(cu, cu.result(), np.arange(0, 2048, 64), oracle.Q_NONE)
    show(capsys, f"attention split3: S {e_s:.3e} (two accumulators {e_sh[0]:.3e} / on load {e_sh[1]:.3e}), "
                 f"O {e_o:.3e} (O without operand scale {e_u:.3e})")
    assert e_s <= TOL["split"] and e_sl <= TOL["split"] and max(e_sh) <= TOL["split"]
    assert e_o <= TOL["split"]
