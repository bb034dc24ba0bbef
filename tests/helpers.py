"""Shared helpers of the GPU parity tests: build stored operands with a given
layout / leading dimension / batch stride from seeded synthetic values, run the
product through the C ABI, and compute the oracle's reference values."""
from __future__ import annotations

import numpy as np

import mixed_precision_matmul_gb300 as mpg
import oracle
import synthetic

SENTINEL_BITS = np.uint32(0x7FC0DEAD)   # a quiet NaN pattern no kernel produces

# oracle quantisation of each precision mode (mode Q)
MODE_Q = {
    mpg.FP16_F32ACC: oracle.Q_FP16,
    mpg.BF16_F32ACC: oracle.Q_BF16,
    mpg.SPLIT_FP16_3CHAIN: oracle.Q_SPLIT3,
    mpg.SPLIT_FP16_1CHAIN: oracle.Q_SPLIT1,
    mpg.FP32_FFMA: oracle.Q_NONE,
    mpg.SPLIT_A_FP16_2CHAIN: oracle.Q_SPLIT3,    # A: hi + lo*2^-11
    mpg.SPLIT_FP16_4CHAIN: oracle.Q_SPLIT4,
}
# quantisation of B where it differs from A's
MODE_QB = {mpg.SPLIT_A_FP16_2CHAIN: oracle.Q_FP16}

TOL = {  # normalised error bars
    "q16": 1e-5,     # fp16 / bf16 against the quantised-input problem
    "tf32": 2e-3,    # tf32 against the fp32-input problem
    "split": 5e-6,   # split hi/lo against the fp32-input problem
}


def torch_dtype(name):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[name]


def dtype_code(name):
    return {"f32": mpg.F32, "f16": mpg.F16, "bf16": mpg.BF16}[name]


def round_to(x: np.ndarray, name: str) -> np.ndarray:
    """Storage rounding of generated fp32 values (input preparation)."""
    if name == "f16":
        return x.astype(np.float16).astype(np.float32)
    if name == "bf16":
        codes = synthetic.bf16_codes_from_f32(x)
        return (codes.astype(np.uint32) << 16).view(np.float32)
    return x.astype(np.float32)


def stored(x: np.ndarray, layout: int, ld: int) -> np.ndarray:
    """(batch, rows, cols) logical values -> (batch, outer, ld) stored buffer."""
    b, rows, cols = x.shape
    if layout == mpg.ROW_MAJOR:
        buf = np.zeros((b, rows, ld), dtype=np.float32)
        buf[:, :, :cols] = x
    else:
        buf = np.zeros((b, cols, ld), dtype=np.float32)
        buf[:, :, :rows] = np.transpose(x, (0, 2, 1))
    return buf


class Case:
    """One product on the GPU, with its inputs kept for the oracle."""

    def __init__(self, m, n, k, mode, batch=1, in_dtype="f32", a_layout=mpg.ROW_MAJOR,
                 b_layout=mpg.ROW_MAJOR, pad=(0, 0, 0), alpha=1.0, beta=0.0, seed=0,
                 dist="uniform", opts=None, a=None, b=None, c0=None):
        import torch
        self.m, self.n, self.k, self.batch, self.mode = m, n, k, batch, mode
        self.alpha, self.beta, self.opts = alpha, beta, opts
        self.a_layout, self.b_layout, self.in_dtype = a_layout, b_layout, in_dtype
        gen = {"uniform": synthetic.uniform, "normal": synthetic.normal,
               "loguniform": synthetic.loguniform_signed, "asym": synthetic.asymmetric}[dist]
        if a is None:
            a = gen((batch, m, k), synthetic.SEED_A + 100 * seed)
        if b is None:
            b = gen((batch, k, n), synthetic.SEED_B + 100 * seed)
        if c0 is None:
            c0 = synthetic.uniform((batch, m, n), synthetic.SEED_C0 + 100 * seed)
        self.a = round_to(np.asarray(a, np.float32).reshape(batch, m, k), in_dtype)
        self.b = round_to(np.asarray(b, np.float32).reshape(batch, k, n), in_dtype)
        self.c0 = np.asarray(c0, np.float32).reshape(batch, m, n)
        pa, pb, pc = pad
        self.lda = (k if a_layout == mpg.ROW_MAJOR else m) + pa
        self.ldb = (n if b_layout == mpg.ROW_MAJOR else k) + pb
        self.ldc = n + pc
        self.lda, self.ldb, self.ldc = max(self.lda, 1), max(self.ldb, 1), max(self.ldc, 1)
        dev = torch.device("cuda")
        td = torch_dtype(in_dtype)
        self.A = torch.from_numpy(stored(self.a, a_layout, self.lda)).to(dev).to(td).contiguous()
        self.B = torch.from_numpy(stored(self.b, b_layout, self.ldb)).to(dev).to(td).contiguous()
        cbuf = np.full((batch, m, self.ldc), 0, dtype=np.float32)
        cbuf.view(np.uint32)[...] = SENTINEL_BITS
        cbuf[:, :, :n] = self.c0
        self.C = torch.from_numpy(cbuf).to(dev)

    def run(self, workspace=None, check=True, stream=0, exact_ws=False):
        """exact_ws: size the workspace with the query that sees the operands
        (it includes aligned copies of operands TMA cannot describe)."""
        import torch
        sa = self.A.stride(0) if self.batch > 1 else 0
        sb = self.B.stride(0) if self.batch > 1 else 0
        if exact_ws:
            ws_bytes = mpg.workspace_size_ex(self.m, self.n, self.k, self.batch, self.A.data_ptr(), self.lda, sa,
                                             dtype_code(self.in_dtype), self.a_layout, self.B.data_ptr(), self.ldb,
                                             sb, dtype_code(self.in_dtype), self.b_layout, self.mode, self.opts)
        else:
            ws_bytes = mpg.workspace_size(self.m, self.n, self.k, self.batch, self.mode, self.opts)
        if workspace is None and ws_bytes:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        wsp = workspace.data_ptr() if workspace is not None else 0
        wsl = workspace.numel() if workspace is not None else 0
        sc = self.C.stride(0) if self.batch > 1 else 0
        st = mpg.gemm_raw(self.m, self.n, self.k, self.batch,
                          self.A.data_ptr(), self.lda, sa, dtype_code(self.in_dtype), self.a_layout,
                          self.B.data_ptr(), self.ldb, sb, dtype_code(self.in_dtype), self.b_layout,
                          self.C.data_ptr(), self.ldc, sc, self.alpha, self.beta, self.mode,
                          wsp, wsl, stream, self.opts, check=check)
        return st

    def result(self) -> np.ndarray:
        import torch
        torch.cuda.synchronize()
        assert mpg.device_status() == mpg.OK, mpg.last_error()
        full = self.C.cpu().numpy()
        pad = full[:, :, self.n:]
        assert np.all(pad.view(np.uint32) == SENTINEL_BITS), "padding of C was written"
        return full[:, :, :self.n].copy()

    # ---- oracle
    def _exps(self):
        if self.opts is None:
            return 0, 0
        return int(self.opts.split_exp_a), int(self.opts.split_exp_b)

    def reference(self, q, batches=None, qb=None):
        """Full-grid oracle (ref, den) per batch for quantisation q (of A and,
        unless qb is given, of B)."""
        sa, sb = self._exps()
        qb = q if qb is None else qb
        out = []
        for bi in (range(self.batch) if batches is None else batches):
            out.append(oracle.gemm(self.a[bi], self.b[bi], self.c0[bi], self.alpha, self.beta,
                                   q, qb, sa, sb))
        return out

    def reference_points(self, q, bi, rows, cols):
        sa, sb = self._exps()
        return oracle.gemm_points(self.a[bi], self.b[bi], self.k, rows, cols, self.c0[bi],
                                  self.alpha, self.beta, q, q, sa, sb)

    def errors(self, C=None, batches=None):
        """(error vs mode R, error vs mode Q) over the listed batches."""
        C = self.result() if C is None else C
        bl = list(range(self.batch)) if batches is None else list(batches)
        eR = eQ = 0.0
        q = MODE_Q.get(self.mode)
        refsR = self.reference(oracle.Q_NONE, bl)
        refsQ = self.reference(q, bl, MODE_QB.get(self.mode)) if q is not None else None
        for i, bi in enumerate(bl):
            eR = max(eR, oracle.max_rel_err(C[bi], *refsR[i]))
            if refsQ is not None:
                eQ = max(eQ, oracle.max_rel_err(C[bi], *refsQ[i]))
        return eR, eQ


def sample_points(m, n, count, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    rows = g.integers(0, m, size=count)
    cols = g.integers(0, n, size=count)
    # always include the corners and the last row/column (tails)
    rows = np.concatenate([rows, [0, 0, m - 1, m - 1]])
    cols = np.concatenate([cols, [0, n - 1, 0, n - 1]])
    return rows.astype(np.int64), cols.astype(np.int64)
