"""Test configuration: markers and import path.

``-m gpu`` tests need a CUDA GPU and the built CUDA library; everything else
runs on the CPU (oracle pins, host-side validation, symbol exports).
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running case")
    config.addinivalue_line("markers", "allow_fault: the test reads and clears the library's device fault bits")
