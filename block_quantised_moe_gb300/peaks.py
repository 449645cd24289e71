"""Measure the tensor-core MMA issue rates the prefill kernels are compared to.

``python -m block_quantised_moe_gb300.peaks`` builds the library if needed and
prints TFLOP/s of back-to-back tcgen05.mma (kind::f16, the block-scaled NVFP4
kind and the block-scaled MX FP8 kind, M=128, N=128/256) on cuda:0 through
``moe_measure_mma_peak``.
"""


def main():
    from . import build
    build.build()
    from . import abi
    for kind, name in ((abi.MOE_PEAK_F16, "kind::f16 M=128 K=16"), (abi.MOE_PEAK_FP4, "kind::mxf4nvf4 M=128 K=64"),
                       (abi.MOE_PEAK_MXFP8, "kind::mxf8f6f4 E4M3 M=128 K=32")):
        for n in (128, 256):
            print(f"{name} N={n}: {abi.moe_measure_mma_peak(kind, n):.1f} TFLOP/s", flush=True)


if __name__ == "__main__":
    main()
