"""ctypes view of the C ABI declared in include/mao.h (argument marshalling only)."""

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))

MAO_OK = 0
MAO_ERR_INVALID_ARG = 1
MAO_ERR_UNSUPPORTED = 2
MAO_ERR_MISALIGNED = 3
MAO_ERR_WORKSPACE = 4
MAO_ERR_CUDA = 5
MAO_ERR_TIMEOUT = 6
MAO_ERR_NUMERIC = 7

MAO_F32 = 0
MAO_BF16 = 1
MAO_I8 = 2      # ns_orthogonalize input only
MAO_SIGN1 = 3   # ns_orthogonalize input only (packed signs, ld == cols)

# every symbol include/mao.h declares
EXPORTS = (
    "mao_abi_version",
    "mao_status_string",
    "muon_momentum_update",
    "ns_workspace_bytes",
    "ns_orthogonalize",
    "muon_step",
    "muon_step_host",
    "sign_muon_step",
    "ns_orthogonalize_noalloc",
    "ns_noalloc_workspace_bytes",
    "ns_blockwise_workspace_bytes",
    "ns_orthogonalize_blockwise",
    "sign_pack_bits",
    "majority_vote_packed",
    "sign_int8",
    "majority_vote_int8",
    "apply_update",
    "dion_workspace_bytes",
    "dion_step",
    "mao_set_wait_limit",
    "mao_get_wait_limit",
    "mao_sync_status",
    "mao_launch_count",
    "mao_profile_begin",
    "mao_profile_span_begin",
    "mao_profile_span_end",
    "mao_profile_end",
    "mao_profile_end_tagged",
)


class MaoMat(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
        ("ld", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class MaoError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        name = _LIB.mao_status_string(status).decode() if _LIB else str(status)
        super().__init__("%s failed: %s" % (fn, name))


_LIB = None


def library_path():
    return os.environ.get("MAO_LIBRARY", os.path.join(_PKG, "libmao.so"))


def load():
    """Load libmao.so (raises if it has not been built: there is no fallback path)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            "libmao.so not found at %s; build it with "
            "`python -m matrix_aware_optimizers_gb300.build`" % path)
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    vp = ctypes.c_void_p
    lib.mao_abi_version.restype = ctypes.c_int32
    lib.mao_abi_version.argtypes = []
    lib.mao_status_string.restype = ctypes.c_char_p
    lib.mao_status_string.argtypes = [ctypes.c_int]
    lib.muon_momentum_update.restype = ctypes.c_int
    lib.muon_momentum_update.argtypes = [P(MaoMat), P(MaoMat), ctypes.c_int32, ctypes.c_float, vp]
    lib.ns_workspace_bytes.restype = ctypes.c_size_t
    lib.ns_workspace_bytes.argtypes = [P(MaoMat), ctypes.c_int32, ctypes.c_int32]
    lib.ns_orthogonalize.restype = ctypes.c_int
    lib.ns_orthogonalize.argtypes = [
        P(MaoMat), P(MaoMat), ctypes.c_int32, ctypes.c_int32, P(ctypes.c_float), ctypes.c_int32,
        ctypes.c_float, ctypes.c_int32, P(ctypes.c_void_p), vp, ctypes.c_size_t, vp]
    lib.muon_step.restype = ctypes.c_int
    lib.muon_step.argtypes = [
        P(MaoMat), P(MaoMat), P(MaoMat), P(MaoMat), ctypes.c_int32, ctypes.c_float, ctypes.c_float,
        ctypes.c_int32, P(ctypes.c_float), ctypes.c_int32, ctypes.c_float, ctypes.c_int32, vp,
        ctypes.c_size_t, vp]
    lib.muon_step_host.restype = ctypes.c_int
    lib.muon_step_host.argtypes = [
        P(MaoMat), P(MaoMat), P(MaoMat), P(MaoMat), ctypes.c_int32, ctypes.c_float, ctypes.c_float,
        ctypes.c_int32, P(ctypes.c_float), ctypes.c_int32, ctypes.c_float, ctypes.c_int32, vp,
        ctypes.c_size_t, vp, vp, ctypes.c_size_t, vp, vp, ctypes.c_size_t, vp, vp, vp]
    lib.sign_muon_step.restype = ctypes.c_int
    lib.sign_muon_step.argtypes = [
        P(MaoMat), P(MaoMat), P(MaoMat), ctypes.c_int32, vp, ctypes.c_int64, vp, ctypes.c_float,
        ctypes.c_float, ctypes.c_int32, P(ctypes.c_float), ctypes.c_int32, ctypes.c_float,
        ctypes.c_int32, vp, ctypes.c_size_t, vp]
    lib.ns_orthogonalize_noalloc.restype = ctypes.c_int
    lib.ns_orthogonalize_noalloc.argtypes = [
        P(MaoMat), P(MaoMat), ctypes.c_int32, ctypes.c_int32, P(ctypes.c_float), ctypes.c_int32,
        ctypes.c_float, ctypes.c_int32, P(ctypes.c_void_p), vp]
    lib.ns_noalloc_workspace_bytes.restype = ctypes.c_size_t
    lib.ns_noalloc_workspace_bytes.argtypes = []
    lib.ns_blockwise_workspace_bytes.restype = ctypes.c_size_t
    lib.ns_blockwise_workspace_bytes.argtypes = [P(MaoMat), ctypes.c_int32, ctypes.c_int64,
                                                 ctypes.c_int64, ctypes.c_int32]
    lib.ns_orthogonalize_blockwise.restype = ctypes.c_int
    lib.ns_orthogonalize_blockwise.argtypes = [
        P(MaoMat), P(MaoMat), ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
        P(ctypes.c_float), ctypes.c_int32, ctypes.c_float, ctypes.c_int32, vp, ctypes.c_size_t, vp]
    lib.sign_pack_bits.restype = ctypes.c_int
    lib.sign_pack_bits.argtypes = [P(MaoMat), vp, vp]
    lib.majority_vote_packed.restype = ctypes.c_int
    lib.majority_vote_packed.argtypes = [vp, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, vp, vp]
    lib.sign_int8.restype = ctypes.c_int
    lib.sign_int8.argtypes = [P(MaoMat), vp, vp]
    lib.majority_vote_int8.restype = ctypes.c_int
    lib.majority_vote_int8.argtypes = [vp, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, vp, vp,
                                       vp, vp]
    lib.apply_update.restype = ctypes.c_int
    lib.apply_update.argtypes = [P(MaoMat), P(ctypes.c_void_p), P(MaoMat), ctypes.c_int32,
                                 ctypes.c_float, vp]
    lib.dion_workspace_bytes.restype = ctypes.c_size_t
    lib.dion_workspace_bytes.argtypes = [P(MaoMat), ctypes.c_int32, ctypes.c_int32]
    lib.dion_step.restype = ctypes.c_int
    lib.dion_step.argtypes = [P(MaoMat), P(MaoMat), P(MaoMat), P(MaoMat), P(MaoMat),
                              P(ctypes.c_void_p),
                              ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                              ctypes.c_int32, vp, ctypes.c_size_t, vp]
    lib.mao_set_wait_limit.restype = None
    lib.mao_set_wait_limit.argtypes = [ctypes.c_uint64]
    lib.mao_get_wait_limit.restype = ctypes.c_uint64
    lib.mao_get_wait_limit.argtypes = []
    lib.mao_sync_status.restype = ctypes.c_int
    lib.mao_sync_status.argtypes = [vp]
    lib.mao_launch_count.restype = ctypes.c_int64
    lib.mao_launch_count.argtypes = []
    lib.mao_profile_begin.restype = ctypes.c_int
    lib.mao_profile_begin.argtypes = [ctypes.c_int32]
    lib.mao_profile_span_begin.restype = ctypes.c_int
    lib.mao_profile_span_begin.argtypes = [ctypes.c_int32]
    lib.mao_profile_span_end.restype = ctypes.c_int32
    lib.mao_profile_span_end.argtypes = [P(ctypes.c_float), ctypes.c_int32]
    lib.mao_profile_end.restype = ctypes.c_int32
    lib.mao_profile_end.argtypes = [P(ctypes.c_float), ctypes.c_int32]
    lib.mao_profile_end_tagged.restype = ctypes.c_int32
    lib.mao_profile_end_tagged.argtypes = [P(ctypes.c_float), P(ctypes.c_int32), ctypes.c_int32]
    _LIB = lib
    return lib


def check(fn, status):
    if status != MAO_OK:
        raise MaoError(fn, status)
