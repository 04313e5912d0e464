"""Shape classes of the configuration table, their representative shapes and candidates.

A class is decided by the operands' TMA alignment and by the grid depth in waves of 128 x 128
tiles at two CTAs per SM on the device's multiprocessors (152 on a GB300, the default here):
the same rule `config_table.h` applies at run time with the count it reads from the device.
The M <= 8 and N <= 8 shapes always take the bandwidth kernels and are not swept."""
from __future__ import annotations

SMS = 152

# class name -> (representative (M, N, K) shapes, candidate configuration names)
ALIGNED = ["dp_tma_128x128_s3", "dp_tma_128x256_s4", "sk_tma_ws_128x128_s3", "sk_tma_ws_128x256_s4",
           "sk_tma_ws_256x128_s4", "pdp_tma_ws_128x256_s4", "sk_tma_ws_128x256_k64_s2",
           "sk_tma_ws_256x128_k64_s2", "splitk_cpasync_64x64", "ck_tma_128x256_k64_s2",
           "ck_tma_256x128_k64_s2", "ck_tma_128x256_s4", "ck_tma_256x128_s4"]
UNALIGNED = ["packed_sk_tma_128x256_s4", "packed_dp_tma_128x128_s3", "packed_sk_tma_256x128_k64_s2",
             "sk_cpasync_128x256_s4",
             "dp_cpasync_128x256_s4", "dp_cpasync_128x128_s3", "splitk_cpasync_64x64",
             "packed_ck_tma_128x256_k64_s2"]

CLASSES = {
    "aligned_tiny": ([(128, 128, 128), (256, 256, 256), (512, 512, 512), (128, 64, 2048)], ALIGNED),
    "aligned_small": ([(1024, 1024, 1024), (1024, 2048, 1024), (2048, 2048, 2048)], ALIGNED),
    "aligned_medium": ([(4096, 4096, 4096), (4096, 3072, 2048), (3072, 4096, 4096)], ALIGNED),
    "aligned_large": ([(8192, 8192, 8192), (16384, 12288, 4096)], ALIGNED),
    "unaligned_tiny": ([(97, 95, 513), (127, 129, 4099), (255, 257, 253), (511, 509, 515)], UNALIGNED),
    "unaligned_small": ([(1001, 999, 1003), (2047, 2045, 2049)], UNALIGNED),
    "unaligned_medium": ([(4095, 3001, 1537), (4097, 4093, 4099)], UNALIGNED),
    "unaligned_large": ([(8191, 8193, 8195)], UNALIGNED),
}

CLASS_ORDER = list(CLASSES)


def waves(M: int, N: int, batch: int = 1, sms: int = SMS) -> float:
    return ((M + 127) // 128) * ((N + 127) // 128) * batch / (2.0 * sms)


def classify(M: int, N: int, aligned: bool, batch: int = 1, sms: int = SMS) -> str:
    """The class of a problem on a part with `sms` multiprocessors (mirrors table_choose in
    config_table.h)."""
    prefix = "aligned" if aligned else "unaligned"
    if M * N * batch <= 512 * 512:
        return prefix + "_tiny"
    w = waves(M, N, batch, sms)
    if w < 1.0:
        return prefix + "_small"
    if w < 6.0:
        return prefix + "_medium"
    return prefix + "_large"


def clusterk_preferred(M: int, N: int, K: int, batch: int = 1, sms: int = SMS) -> bool:
    """Grids that take the cluster split-K kernel ahead of the class table (mirrors
    clusterk_preferred in config_table.h): more than 512 x 512 outputs, at most sms / 4 tiles
    of 128 x 256, at least four 64-wide k-tiles."""
    if M * N * batch <= 512 * 512:
        return False
    tiles = ((M + 127) // 128) * ((N + 255) // 256) * batch
    return tiles * 4 <= sms and (K + 63) // 64 >= 4


def expected_config(M: int, N: int, K: int, aligned: bool, winners: dict, batch: int = 1,
                    sms: int = SMS) -> str:
    """The configuration the library picks for a non-skinny problem: the cluster split-K
    kernel where clusterk_preferred holds, else the class's measured winner."""
    if clusterk_preferred(M, N, K, batch, sms):
        return "ck_tma_128x256_s4" if aligned else "packed_ck_tma_128x256_k64_s2"
    return winners[classify(M, N, aligned, batch, sms)]
