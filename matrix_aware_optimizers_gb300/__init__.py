"""GB300 (sm_103a) Muon / Sign-Muon optimizer step behind a C ABI (libmao.so).

This module only marshals PyTorch CUDA tensors into the C ABI of include/mao.h;
every stage of the step runs in the library's CUDA kernels. There is no CPU or
PyTorch fallback: if libmao.so is missing, the calls raise.

Functions (same names as the C ABI):
  muon_momentum_update(M, G, mu)                     M <- mu*M + G
  ns_workspace_bytes(X, compute)                     workspace size for ns_orthogonalize
  ns_orthogonalize(inp, out, steps, coeffs, ...)     Newton–Schulz polar factor (+ packed signs)
  muon_step(W, M, G, mu, lr, ...)                    momentum + Newton–Schulz + update, fused
  muon_step_host(W, M, G, mu, lr, g_host, ...)      muon_step with host gradients / weights
  sign_muon_step(W, M, G, words, vote, mu, lr, ...)  momentum + NS signs + vote + update
  ns_orthogonalize_blockwise(inp, out, block, ...)   Newton–Schulz of every block on its own
  sign_pack_bits(U, bits)                            sign + 1-bit pack
  majority_vote_packed(bits, nbits, vote)            vote over workers' packed signs
  sign_int8(U, s)                                    sign as int8 +-1 (all-reduce variant)
  majority_vote_int8(s, n, sum, s_bar, vote)         int8 SUM over workers + threshold
  apply_update(W, lr, vote=..., U=...)               W <- W - lr*D
  dion_step(X, M, G, Q, mu, lr, ...)                 one Dion step (low-rank, error feedback)
  sync_status()                                      stream sync + device error word
"""

import ctypes

import torch

from . import _abi
from ._abi import MaoError  # noqa: F401

# Default Newton–Schulz coefficients (a, b, c): the quintic used by Muon.
QUINTIC = (3.4445, -4.7750, 2.0315)

_DT = {torch.float32: _abi.MAO_F32, torch.bfloat16: _abi.MAO_BF16, torch.int8: _abi.MAO_I8}
_COMPUTE = {"f32": _abi.MAO_F32, "bf16": _abi.MAO_BF16,
            torch.float32: _abi.MAO_F32, torch.bfloat16: _abi.MAO_BF16}


def lib():
    return _abi.load()


def _as_list(x):
    if x is None:
        return None
    return list(x) if isinstance(x, (list, tuple)) else [x]


class PackedSigns:
    """A rows x cols sign matrix held as packed words (int32 tensor of ceil(rows*cols/32)
    words, header layout), usable as an ns_orthogonalize input."""

    def __init__(self, words, rows, cols):
        if not words.is_cuda or words.dtype != torch.int32 or not words.is_contiguous():
            raise ValueError("words must be a contiguous int32 CUDA tensor")
        if words.numel() < packed_words(rows, cols):
            raise ValueError("too few words for a %d x %d sign matrix" % (rows, cols))
        self.words, self.shape = words, (int(rows), int(cols))
        self.device = words.device


def _mat(t, allow_none=False, like=None):
    if isinstance(t, PackedSigns):
        R, C = t.shape
        return _abi.MaoMat(t.words.data_ptr(), R, C, C, _abi.MAO_SIGN1, 0)
    if t is None:
        if not allow_none:
            raise ValueError("tensor required")
        return _abi.MaoMat(None, like.shape[0], like.shape[1], like.shape[1], _abi.MAO_F32, 0)
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit column stride")
    if t.dtype not in _DT:
        raise ValueError("dtype must be float32, bfloat16 or int8")
    return _abi.MaoMat(t.data_ptr(), t.shape[0], t.shape[1], max(t.stride(0), t.shape[1]),
                       _DT[t.dtype], 0)


def _mats(ts, allow_none=False, like=None):
    arr = (_abi.MaoMat * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _mat(t, allow_none, like[i] if like is not None else None)
    return arr


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def muon_momentum_update(M, G, mu, stream=None):
    """M <- mu*M + G for each (M, G) pair (one fp32 FMA per element, rounded to M's dtype)."""
    Ms, Gs = _as_list(M), _as_list(G)
    st = lib().muon_momentum_update(_mats(Ms), _mats(Gs), len(Ms), float(mu), _stream(stream))
    _abi.check("muon_momentum_update", st)


def ns_workspace_bytes(X, compute="bf16"):
    Xs = _as_list(X)
    arr = (_abi.MaoMat * len(Xs))()
    for i, x in enumerate(Xs):
        shape = x.shape if hasattr(x, "shape") else x
        arr[i] = _abi.MaoMat(None, shape[0], shape[1], shape[1], _abi.MAO_F32, 0)
    n = lib().ns_workspace_bytes(arr, len(Xs), _COMPUTE[compute])
    if n == 0:
        raise ValueError("invalid shapes for ns_workspace_bytes")
    return int(n)


def workspace(X, compute="bf16", device=None):
    """A device buffer of ns_workspace_bytes(X) bytes (256-byte aligned by the allocator)."""
    n = ns_workspace_bytes(X, compute)
    dev = device if device is not None else torch.device("cuda")
    return torch.empty(n, dtype=torch.uint8, device=dev)


def ns_orthogonalize(inp, out, steps=5, coeffs=QUINTIC, eps=1e-7, compute="bf16",
                     sign_bits=None, ws=None, stream=None):
    """Newton–Schulz orthogonalisation of each input into out (and/or packed signs).

    coeffs: one (a, b, c) triple for every step, or a list of `steps` triples.
    out entries may be None when sign_bits (int32 tensors of ceil(R*C/32) words) are given.
    """
    ins = _as_list(inp)
    outs = _as_list(out) if out is not None else [None] * len(ins)
    co = list(coeffs)
    if len(co) == 3 and not isinstance(co[0], (list, tuple)):
        flat, stride = [float(c) for c in co], 0
    else:
        if len(co) != steps:
            raise ValueError("need one coefficient triple per step")
        flat, stride = [float(c) for t in co for c in t], 3
    carr = (ctypes.c_float * len(flat))(*flat)
    bits = _as_list(sign_bits)
    barr = None
    if bits is not None:
        barr = (ctypes.c_void_p * len(bits))(*[b.data_ptr() if b is not None else None for b in bits])
    if ws is None:
        ws = workspace(ins, compute, ins[0].device)
    st = lib().ns_orthogonalize(
        _mats(ins), _mats(outs, allow_none=True, like=ins), len(ins), int(steps), carr, stride,
        float(eps), _COMPUTE[compute], barr, ctypes.c_void_p(ws.data_ptr()), ws.numel(),
        _stream(stream))
    _abi.check("ns_orthogonalize", st)


def muon_step(W, M, G, mu, lr, steps=5, coeffs=QUINTIC, eps=1e-7, compute="bf16", ws=None,
              W_out=None, stream=None):
    """One whole Muon step: M <- mu*M + G, U = Newton-Schulz(M), W' = W - lr*U into W_out
    (W itself when W_out is None).

    U is never stored: the last product updates W from U's fp32 values. The workspace is
    that of ns_orthogonalize(M) (workspace(M, "bf16", device)).
    """
    Ws, Ms, Gs = _as_list(W), _as_list(M), _as_list(G)
    Wo = _as_list(W_out) if W_out is not None else None
    if not (len(Ws) == len(Ms) == len(Gs)) or (Wo is not None and len(Wo) != len(Ws)):
        raise ValueError("W, M, G (and W_out) need the same number of matrices")
    carr, stride = _coeff_args(coeffs, steps)
    if ws is None:
        ws = workspace(Ms, compute, Ms[0].device)
    st = lib().muon_step(_mats(Ws), _mats(Ms), _mats(Gs), _mats(Wo) if Wo is not None else None,
                         len(Ws), float(mu), float(lr),
                         int(steps), carr, stride, float(eps), _COMPUTE[compute],
                         ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(stream))
    _abi.check("muon_step", st)


def muon_step_host(W, M, G, mu, lr, g_host, g_dev, w_host, w_dev, steps=5, coeffs=QUINTIC,
                   eps=1e-7, compute="bf16", ws=None, W_out=None, stream=None, wait_event=None,
                   record_event=None):
    """muon_step with host data: g_host (pinned CPU tensor) is copied into g_dev (the device
    tensor whose storage holds G) before the step, and w_dev (the device tensor holding the
    new weights) into w_host (pinned CPU tensor) after it, all on `stream`; wait_event /
    record_event (torch.cuda.Event) order the step's compute across streams."""
    Ws, Ms, Gs = _as_list(W), _as_list(M), _as_list(G)
    Wo = _as_list(W_out) if W_out is not None else None
    if g_host.is_cuda or w_host.is_cuda or not g_dev.is_cuda or not w_dev.is_cuda:
        raise ValueError("g_host / w_host must be host tensors and g_dev / w_dev device tensors")
    gb = g_host.numel() * g_host.element_size()
    wb = w_dev.numel() * w_dev.element_size()
    if g_dev.numel() * g_dev.element_size() != gb or w_host.numel() * w_host.element_size() != wb:
        raise ValueError("host and device buffers of different sizes")
    carr, stride = _coeff_args(coeffs, steps)
    if ws is None:
        ws = workspace(Ms, compute, Ms[0].device)
    if record_event is not None and not record_event.cuda_event:
        record_event.record(stream)  # a torch event exists only once recorded
    ev = lambda e: ctypes.c_void_p(e.cuda_event if e is not None else None)  # noqa: E731
    st = lib().muon_step_host(
        _mats(Ws), _mats(Ms), _mats(Gs), _mats(Wo) if Wo is not None else None, len(Ws),
        float(mu), float(lr), int(steps), carr, stride, float(eps), _COMPUTE[compute],
        ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(g_host.data_ptr()),
        ctypes.c_void_p(g_dev.data_ptr()), gb, ctypes.c_void_p(w_host.data_ptr()),
        ctypes.c_void_p(w_dev.data_ptr()), wb, _stream(stream), ev(wait_event), ev(record_event))
    _abi.check("muon_step_host", st)


class PreparedCall:
    """A library call whose arguments were marshalled once: calling the object repeats the
    call with the same tensors (which must keep their storage), scalars and stream. For
    training loops whose step is short enough that building the arguments on the host each
    time would cost more than the GPU work."""

    def __init__(self, name, args, keep):
        self._fn = getattr(lib(), name)
        self._name = name
        self._args = args
        self._keep = keep  # the tensors and ctypes objects the arguments point into

    def __call__(self):
        _abi.check(self._name, self._fn(*self._args))


def sign_muon_step(W, M, G, words, vote, mu, lr, steps=5, coeffs=QUINTIC, eps=1e-7,
                   compute="bf16", ws=None, stream=None, prepare=False):
    """One whole Sign-Muon step: momentum of every worker, Newton-Schulz with the packed
    signs into words[m] (int32 tensor [W_n][stride]), the majority vote into `vote` and
    W <- W - lr * vote; the same results as the four separate calls. With prepare=True the
    call is not made: a PreparedCall that makes it (on `stream`, or the stream current now)
    is returned."""
    Ms, Gs = _as_list(M), _as_list(G)
    if len(Ms) != len(Gs) or words.dim() != 2 or words.shape[0] != len(Ms) or \
            words.stride(1) != 1 or words.dtype != torch.int32:
        raise ValueError("need one M and G per worker and int32 words [W_n][stride]")
    carr, stride = _coeff_args(coeffs, steps)
    if ws is None:
        ws = workspace(Ms, compute, Ms[0].device)
    wm, ma, ga = _mat(W), _mats(Ms), _mats(Gs)
    args = (ctypes.byref(wm), ma, ga, len(Ms), ctypes.c_void_p(words.data_ptr()), words.stride(0),
            ctypes.c_void_p(vote.data_ptr()), float(mu), float(lr), int(steps), carr, stride,
            float(eps), _COMPUTE[compute], ctypes.c_void_p(ws.data_ptr()), ws.numel(),
            _stream(stream))
    if prepare:
        return PreparedCall("sign_muon_step", args, (W, Ms, Gs, words, vote, ws, wm, ma, ga, carr))
    _abi.check("sign_muon_step", lib().sign_muon_step(*args))


def _coeff_args(coeffs, steps):
    co = list(coeffs)
    if len(co) == 3 and not isinstance(co[0], (list, tuple)):
        flat, stride = [float(c) for c in co], 0
    else:
        if len(co) != steps:
            raise ValueError("need one coefficient triple per step")
        flat, stride = [float(c) for t in co for c in t], 3
    return (ctypes.c_float * len(flat))(*flat), stride


def ns_blockwise_workspace_bytes(X, block, compute="bf16"):
    Xs = _as_list(X)
    arr = (_abi.MaoMat * len(Xs))()
    for i, x in enumerate(Xs):
        shape = x.shape if hasattr(x, "shape") else x
        arr[i] = _abi.MaoMat(None, shape[0], shape[1], shape[1], _abi.MAO_F32, 0)
    n = lib().ns_blockwise_workspace_bytes(arr, len(Xs), int(block[0]), int(block[1]),
                                           _COMPUTE[compute])
    if n == 0:
        raise ValueError("invalid shapes or block for ns_blockwise_workspace_bytes")
    return int(n)


def ns_orthogonalize_blockwise(inp, out, block, steps=5, coeffs=QUINTIC, eps=1e-7,
                               compute="bf16", ws=None, stream=None):
    """Newton–Schulz of every (block[0] x block[1]) block of each input on its own."""
    ins, outs = _as_list(inp), _as_list(out)
    carr, stride = _coeff_args(coeffs, steps)
    if ws is None:
        n = ns_blockwise_workspace_bytes(ins, block, compute)
        ws = torch.empty(n, dtype=torch.uint8, device=ins[0].device)
    st = lib().ns_orthogonalize_blockwise(
        _mats(ins), _mats(outs), len(ins), int(block[0]), int(block[1]), int(steps), carr, stride,
        float(eps), _COMPUTE[compute], ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(stream))
    _abi.check("ns_orthogonalize_blockwise", st)


def packed_words(rows, cols):
    return (rows * cols + 31) // 32


def sign_pack_bits(U, bits=None, stream=None):
    if bits is None:
        bits = torch.empty(packed_words(*U.shape), dtype=torch.int32, device=U.device)
    st = lib().sign_pack_bits(ctypes.byref(_mat(U)), ctypes.c_void_p(bits.data_ptr()), _stream(stream))
    _abi.check("sign_pack_bits", st)
    return bits


def majority_vote_packed(bits, nbits, vote=None, stream=None):
    """bits: int32 tensor [W_n][stride] of packed worker signs; returns the packed vote."""
    if bits.dim() != 2 or bits.stride(1) != 1:
        raise ValueError("bits must be [n_workers][stride] with unit stride")
    if vote is None:
        vote = torch.empty((nbits + 31) // 32, dtype=torch.int32, device=bits.device)
    st = lib().majority_vote_packed(ctypes.c_void_p(bits.data_ptr()), bits.shape[0], bits.stride(0),
                                    int(nbits), ctypes.c_void_p(vote.data_ptr()), _stream(stream))
    _abi.check("majority_vote_packed", st)
    return vote


def sign_int8(U, s=None, stream=None):
    """int8 signs of U (-1 where U < 0, else +1), row-major R x C."""
    if s is None:
        s = torch.empty(U.shape, dtype=torch.int8, device=U.device)
    st = lib().sign_int8(ctypes.byref(_mat(U)), ctypes.c_void_p(s.data_ptr()), _stream(stream))
    _abi.check("sign_int8", st)
    return s


def majority_vote_int8(s, n, sum=None, s_bar=None, vote=None, stream=None):
    """Integer SUM of workers' int8 signs, then the threshold vote.

    s: int8 tensor [W_n][stride] (stride >= n, unit inner stride). Each of sum / s_bar
    (int8, n entries) and vote (int32, ceil(n/32) words) is a tensor to fill, True to
    allocate, or None to skip. Returns (sum, s_bar, vote).
    """
    if s.dim() != 2 or s.stride(1) != 1 or s.dtype != torch.int8:
        raise ValueError("s must be an int8 [n_workers][stride] tensor with unit stride")

    def alloc(x, count, dt):
        if x is True:
            return torch.empty(count, dtype=dt, device=s.device)
        return x if x is not None and x is not False else None

    sum = alloc(sum, n, torch.int8)
    s_bar = alloc(s_bar, n, torch.int8)
    vote = alloc(vote, packed_words(1, n), torch.int32)
    ptr = lambda x: ctypes.c_void_p(x.data_ptr() if x is not None else None)  # noqa: E731
    st = lib().majority_vote_int8(ptr(s), s.shape[0], s.stride(0), int(n), ptr(sum), ptr(s_bar),
                                  ptr(vote), _stream(stream))
    _abi.check("majority_vote_int8", st)
    return sum, s_bar, vote


def apply_update(W, lr, vote=None, U=None, stream=None):
    """W <- W - lr*D with D the packed vote (+1/-1) or the matrix U."""
    Ws = _as_list(W)
    varr = None
    uarr = None
    if vote is not None:
        vs = _as_list(vote)
        varr = (ctypes.c_void_p * len(vs))(*[v.data_ptr() for v in vs])
    if U is not None:
        uarr = _mats(_as_list(U))
    st = lib().apply_update(_mats(Ws), varr, uarr, len(Ws), float(lr), _stream(stream))
    _abi.check("apply_update", st)


def dion_workspace_bytes(shapes, rank):
    """Workspace bytes of one dion_step call over matrices of the given (m, n) shapes."""
    arr = (_abi.MaoMat * len(shapes))()
    for i, sh in enumerate(shapes):
        arr[i] = _abi.MaoMat(None, sh[0], sh[1], sh[1], _abi.MAO_F32, 0)
    n = lib().dion_workspace_bytes(arr, len(shapes), int(rank))
    if n == 0:
        raise ValueError("invalid shapes or rank for dion_workspace_bytes")
    return int(n)


def _q_mat(q):
    if not q.is_cuda or q.dtype != torch.float32 or q.dim() != 2 or q.stride(1) != 1:
        raise ValueError("Q must be a 2-D float32 CUDA tensor with unit column stride")
    return _abi.MaoMat(q.data_ptr(), q.shape[0], q.shape[1], max(q.stride(0), q.shape[1]),
                       _abi.MAO_F32, 0)


def dion_step(X, M, G, Q, mu, lr, P_out=None, ws=None, stream=None, X_out=None):
    """One Dion step for each (X, M, G, Q), any mix of shapes, one rank: X and M updated in
    place, Q replaced by the new right factor (n x r, float32). P_out: optional float32
    tensors (m x r, contiguous) receiving the final P. X_out: optional tensors of X's shapes
    and dtypes receiving the new X (X is then only read)."""
    Xs, Ms, Gs, Qs = _as_list(X), _as_list(M), _as_list(G), _as_list(Q)
    rank = Qs[0].shape[1]
    if any(q.shape[1] != rank for q in Qs):
        raise ValueError("one rank per call")
    qarr = (_abi.MaoMat * len(Qs))()
    for k, q in enumerate(Qs):
        qarr[k] = _q_mat(q)
    parr = None
    if P_out is not None:
        Ps = _as_list(P_out)
        parr = (ctypes.c_void_p * len(Ps))(*[p.data_ptr() if p is not None else None for p in Ps])
    if ws is None:
        ws = torch.empty(dion_workspace_bytes([tuple(x.shape) for x in Xs], rank),
                         dtype=torch.uint8, device=Xs[0].device)
    xo = None
    if X_out is not None:
        Xos = _as_list(X_out)
        if len(Xos) != len(Xs):
            raise ValueError("X_out needs one tensor per X")
        xo = _mats(Xos)
    st = lib().dion_step(_mats(Xs), _mats(Ms), _mats(Gs), qarr, xo, parr, len(Xs), int(rank),
                         float(mu), float(lr), _abi.MAO_BF16, ctypes.c_void_p(ws.data_ptr()),
                         ws.numel(), _stream(stream))
    _abi.check("dion_step", st)


def set_wait_limit(ns):
    """Bound (ns) of every device-side wait of the tensor-core kernels; 0 gives up at once."""
    lib().mao_set_wait_limit(int(ns))


def get_wait_limit():
    return int(lib().mao_get_wait_limit())


def sync_status(stream=None):
    st = lib().mao_sync_status(_stream(stream))
    _abi.check("mao_sync_status", st)


def launch_count():
    """Kernels libmao has launched in this process."""
    return int(lib().mao_launch_count())


PROFILE_TAGS = {0: "tc", 1: "dion_setup", 2: "dion_stage", 3: "dion_gram", 4: "dion_chol",
                5: "dion_split", 6: "dion_norm", 7: "ns_small"}


def profile_begin(max_launches):
    """Record CUDA events around each tensor-core product launch and each Dion CUDA-core
    kernel launch (benchmarking)."""
    _abi.check("mao_profile_begin", lib().mao_profile_begin(int(max_launches)))


def profile_end(max_out=1 << 20):
    """Stop recording; returns the per-launch durations in milliseconds."""
    buf = (ctypes.c_float * max_out)()
    n = lib().mao_profile_end(buf, max_out)
    if n < 0:
        raise MaoError("mao_profile_end", _abi.MAO_ERR_CUDA)
    return [buf[i] for i in range(min(n, max_out))]


def profile_end_tagged(max_out=1 << 20):
    """Stop recording; returns (milliseconds, tag name) per recorded launch."""
    buf = (ctypes.c_float * max_out)()
    tags = (ctypes.c_int32 * max_out)()
    n = lib().mao_profile_end_tagged(buf, tags, max_out)
    if n < 0:
        raise MaoError("mao_profile_end_tagged", _abi.MAO_ERR_CUDA)
    return [(buf[i], PROFILE_TAGS.get(tags[i], str(tags[i]))) for i in range(min(n, max_out))]


def profile_span_begin(max_spans):
    """Record one CUDA event pair around each Newton–Schulz call's run of tensor-core products
    (benchmarking; the products keep overlapping one another's set-up)."""
    _abi.check("mao_profile_span_begin", lib().mao_profile_span_begin(int(max_spans)))


def profile_span_end(max_out=1 << 16):
    """Stop recording; returns the recorded spans in milliseconds."""
    buf = (ctypes.c_float * max_out)()
    n = lib().mao_profile_span_end(buf, max_out)
    if n < 0:
        raise MaoError("mao_profile_span_end", _abi.MAO_ERR_CUDA)
    return [buf[i] for i in range(min(n, max_out))]
