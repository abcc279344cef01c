"""CPU oracle for the GPT-2 training step (test infrastructure only).

Only tests/, the package smoke check and the benchmark's CPU-baseline leg may
import anything under this directory.
"""
